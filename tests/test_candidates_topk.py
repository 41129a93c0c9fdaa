"""kv_attend_candidates_topk against the oracle: exact top-k inside each
row's candidate list (MiniCPM study, section 6), then exact attention over
the kept keys. The kept set is an integer decision taken from fp32 scores on
the GPU and fp64 scores in the oracle, so where the two sets differ the
differing keys must score within rounding of the k-th kept score; the output
is then compared with the oracle's attention over the GPU's own set."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_sparse_kv_gb300 import synth

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


@pytest.mark.parametrize("b,hkv,d,n,recent,c,top_k", [
    (2, 2, 128, 4096, 128, 256, 32),   # the pages' C = 256 -> top-32 on the decode cache
    (1, 2, 128, 1000, 0, 96, 32),      # all int4
    (1, 1, 64, 700, 700, 130, 17),     # all window, C not a power of two
    (2, 1, 32, 300, 40, 64, 64),       # keep everything
])
def test_topk_inside_candidates_matches_oracle(kvq, b, hkv, d, n, recent, c, top_k):
    hq = 8 * hkv if d == 128 else 2 * hkv
    rng = np.random.default_rng(n + c)
    q = O.round_to_bf16(rng.standard_normal((b, hq, 2, d)).astype(np.float32))
    k = O.round_to_bf16(rng.standard_normal((b, hkv, n, d)).astype(np.float32))
    v = O.round_to_bf16(rng.standard_normal((b, hkv, n, d)).astype(np.float32))
    idx = np.stack([np.stack([np.stack([rng.choice(n, c, replace=False) for _ in range(2)])
                              for _ in range(hq)]) for _ in range(b)]).astype(np.int32)
    dev = lambda x: torch.from_numpy(x).cuda().to(torch.bfloat16)  # noqa: E731
    cache = kvq.pack(dev(k), dev(v), recent, "bf16")
    out, sel, status = kvq.attend_candidates_topk(cache, dev(q), torch.from_numpy(idx).cuda(),
                                                  top_k, out_dtype="f32")
    assert kvq.read_status(status) == 0
    packed = O.pack(k, v, recent, "bf16")
    sel = sel.cpu().numpy()
    got = to_np(out)
    for bi in range(b):
        for h in range(hq):
            kh, vh = O.dequantize_head(packed[bi][h // (hq // hkv)])
            keep, scores = O.candidate_topk_select(q[bi, h], kh, idx[bi, h], top_k)
            for i in range(2):
                s = dict(zip(idx[bi, h, i].tolist(), scores[i].tolist()))
                kth = s[int(keep[i, -1])]
                g = set(sel[bi, h, i].tolist())
                assert len(g) == top_k and g <= set(s)
                for t in g ^ set(keep[i].tolist()):
                    assert abs(s[t] - kth) < 1e-4, (t, s[t], kth)
                # scores come out in descending order
                assert all(s[x] >= s[y] - 1e-4 for x, y in zip(sel[bi, h, i], sel[bi, h, i][1:]))
            ref = O.candidate_attention(q[bi, h], kh, vh, sel[bi, h])
            assert O.rel_l2(got[bi, h], ref) <= 1e-4


def test_topk_of_all_keys_is_plain_candidate_attention(kvq):
    rng = np.random.default_rng(3)
    n, d = 500, 128
    q = O.round_to_bf16(rng.standard_normal((1, 16, 1, d)).astype(np.float32))
    k = O.round_to_bf16(rng.standard_normal((1, 2, n, d)).astype(np.float32))
    v = O.round_to_bf16(rng.standard_normal((1, 2, n, d)).astype(np.float32))
    idx = synth.candidate_indices(4, 1, 16, n, 96)
    dev = lambda x: torch.from_numpy(x).cuda().to(torch.bfloat16)  # noqa: E731
    cache = kvq.pack(dev(k), dev(v), 128, "bf16")
    a, _, _ = kvq.attend_candidates_topk(cache, dev(q), torch.from_numpy(idx).cuda(), 96,
                                         out_dtype="f32")
    b, _ = kvq.attend_candidates(cache, dev(q), torch.from_numpy(idx).cuda(), out_dtype="f32")
    # the top-k path is fp32 throughout; plain candidate attention at this
    # shape runs on bf16 tensor-core operands (the bf16 tolerance)
    ref = O.attend_candidates(q, O.pack(k, v, 128, "bf16"), idx)
    assert O.rel_l2(to_np(a), ref) <= 1e-5
    assert O.rel_l2(to_np(b), ref) <= 1e-2
    assert O.rel_l2(to_np(a), to_np(b)) <= 1e-2
