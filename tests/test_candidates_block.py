"""kv_attend_candidates_block: candidate prefill with one list per block of
query rows, against the oracle's candidate attention with every row given its
block's list. The tensor-core path gathers the listed rows once into bf16, so
it is compared with the oracle over bf16-rounded keys and values as well as
the exact ones; the fp32 path is compared at fp32 precision."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from quantized_sparse_kv_gb300 import kvq as k
    k.load_library()
    return k


def to_np(t):
    return t.detach().float().cpu().numpy()


def case(seed, b, hkv, hq, n, d, n_q, block_q, c):
    rng = np.random.default_rng(seed)
    q = O.round_to_bf16(rng.standard_normal((b, hq, n_q, d)).astype(np.float32))
    k = O.round_to_bf16(rng.standard_normal((b, hkv, n, d)).astype(np.float32))
    v = O.round_to_bf16(rng.standard_normal((b, hkv, n, d)).astype(np.float32))
    nb = -(-n_q // block_q)
    idx = np.stack([np.stack([np.stack([rng.choice(n, c, replace=False) for _ in range(nb)])
                              for _ in range(hq)]) for _ in range(b)]).astype(np.int32)
    return q, k, v, idx


def reference(q, k, v, recent, idx, block_q, bf16_rows):
    b, hq, n_q, d = q.shape
    hkv = k.shape[1]
    packed = O.pack(k, v, recent, "bf16")
    out = np.empty(q.shape)
    for bi in range(b):
        for h in range(hq):
            kh, vh = O.dequantize_head(packed[bi][h // (hq // hkv)])
            if bf16_rows:
                kh, vh = O.round_to_bf16(kh), O.round_to_bf16(vh)
            rows = idx[bi, h][np.arange(n_q) // block_q]
            out[bi, h] = O.candidate_attention(q[bi, h], kh, vh, rows)
    return out


@pytest.mark.parametrize("b,hkv,hq,n,recent,n_q,block_q,c", [
    (1, 2, 4, 4096, 128, 300, 128, 256),   # three lists per head, the last block ragged
    (2, 1, 2, 1000, 0, 256, 256, 100),     # two query tiles per list, a partial key tile
    (1, 2, 2, 700, 700, 130, 128, 33),     # all window
])
def test_block_lists_on_the_tensor_cores(kvq, b, hkv, hq, n, recent, n_q, block_q, c):
    q, k, v, idx = case(n + c, b, hkv, hq, n, 128, n_q, block_q, c)
    dev = lambda x: torch.from_numpy(x).cuda().to(torch.bfloat16)  # noqa: E731
    cache = kvq.pack(dev(k), dev(v), recent, "bf16")
    a = kvq.AttendCandidatesBlock(cache, dev(q), torch.from_numpy(idx).cuda(), block_q,
                                  out_dtype="f32")
    a.run()
    assert a.path == "candidates_block_tensor"
    assert kvq.read_status(a.status) == 0
    got = to_np(a.out)
    assert O.rel_l2(got, reference(q, k, v, recent, idx, block_q, False)) <= 1e-2
    assert O.rel_l2(got, reference(q, k, v, recent, idx, block_q, True)) <= 1e-2


@pytest.mark.parametrize("d,block_q,q_dtype", [(64, 50, "bf16"), (128, 100, "bf16"),
                                               (128, 128, "f32")])
def test_block_lists_on_the_fp32_kernel(kvq, d, block_q, q_dtype):
    b, hkv, hq, n, recent, n_q, c = 1, 1, 2, 600, 64, 230, 48
    q, k, v, idx = case(d + block_q, b, hkv, hq, n, d, n_q, block_q, c)
    dev = lambda x: torch.from_numpy(x).cuda().to(torch.bfloat16)  # noqa: E731
    cache = kvq.pack(dev(k), dev(v), recent, "bf16")
    qd = dev(q) if q_dtype == "bf16" else torch.from_numpy(q).cuda()
    a = kvq.AttendCandidatesBlock(cache, qd, torch.from_numpy(idx).cuda(), block_q,
                                  out_dtype="f32")
    a.run()
    assert a.path == "candidates_block"
    assert O.rel_l2(to_np(a.out), reference(q, k, v, recent, idx, block_q, False)) <= 1e-5
