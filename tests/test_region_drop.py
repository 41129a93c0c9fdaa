"""kv_attend_region_drop: the Catnip study's local output ablation (drop sink,
drop recent, drop all history, renormalise P) against the oracle's attention
over the kept keys, and the ablation's output change (relative L2, cosine)
against the oracle's."""
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


@pytest.mark.parametrize("drop", [[0], [1], [0, 1], [2]])
def test_region_drop_small(kvq, drop):
    # [sink | recent | current] on a small chunk, int4 history + bf16 window
    rng = np.random.default_rng(40 + sum(drop))
    bounds, recent = [0, 150, 420, 700], 280
    q = O.round_to_bf16(rng.standard_normal((1, 4, 200, 128)).astype(np.float32))
    k = O.round_to_bf16(rng.standard_normal((1, 2, 700, 128)).astype(np.float32))
    v = O.round_to_bf16(rng.standard_normal((1, 2, 700, 128)).astype(np.float32))
    dev = lambda x: torch.from_numpy(x).cuda().to(torch.bfloat16)  # noqa: E731
    cache = kvq.pack(dev(k), dev(v), recent, "bf16")
    a = kvq.AttendRegionDrop(cache, dev(q), bounds, drop, out_dtype="f32")
    got = to_np(a.run())
    keep = O.region_drop_keys(bounds, drop)
    packed = O.pack(k, v, recent, "bf16")
    for h in range(4):
        kh, vh = O.dequantize_head(packed[0][h // 2])
        ref = O.candidate_attention(q[0, h], kh, vh, np.tile(keep, (200, 1)))
        assert O.rel_l2(got[0, h], ref) <= 1e-2


def test_region_drop_ablation_on_the_video_chunk(kvq):
    bounds = list(synth.CHUNK_REGION_BOUNDS)
    q, k, v = synth.chunk_inputs_torch(17, "cuda", concentrated=4.0)
    n = bounds[-1]
    cache = kvq.pack(k, v, n, "bf16")
    full = to_np(kvq.attend(cache, q, out_dtype="f32")[0])
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    for drop in ([0], [1], [0, 1]):   # sink, recent, all history
        got = to_np(kvq.AttendRegionDrop(cache, q, bounds, drop, out_dtype="f32").run())
        keep = O.region_drop_keys(bounds, drop)
        for h in (3, 20):
            ref_full, _, _ = O.attention(qn[0, h], kn[0, h], vn[0, h])
            ref = O.candidate_attention(qn[0, h], kn[0, h], vn[0, h],
                                        np.tile(keep, (qn.shape[2], 1)))
            assert O.rel_l2(got[0, h], ref) <= 1e-2
            rel, cos = O.output_change(got[0, h], full[0, h])
            rel_ref, cos_ref = O.output_change(ref, ref_full)
            np.testing.assert_allclose(rel, rel_ref, atol=2e-2)
            np.testing.assert_allclose(cos, cos_ref, atol=2e-2)
