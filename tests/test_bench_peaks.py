"""The bench's roofline denominators (CPU): each key format's tensor bound
uses the rate of the MMA its logits kernel issues, and the algorithmic bytes
follow the page layouts."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def test_tensor_peak_per_key_format():
    fp8, bf16 = 4000.0, 1900.0
    # FP8 keys: the e4m3 GEMM figure, with its own source string
    assert bench.tensor_peak(W.KV_FP8, fp8, "fp8 src", bf16) == (fp8, "fp8 src")
    # FP4 keys are converted to f16 tiles (kind::f16): the bf16 rate
    tf, src = bench.tensor_peak(W.KV_FP4, fp8, "fp8 src", bf16)
    assert tf == bf16 and "bf16" in src
    # MXFP4 runs block-scaled kind::mxf4: the FP8 figure times the fp4:fp8 ratio
    tf, src = bench.tensor_peak(W.KV_MXFP4, fp8, "fp8 src", bf16)
    assert tf == fp8 * bench.FP4_PER_FP8 and "ratio" in src
    assert bench.FP4_PER_FP8 == 3.0


def test_algorithmic_bytes_per_token():
    """Key bytes a token: FP8 8192/64 + 4, FP4 64 + 8 + 4, MXFP4 64 + 4."""
    for fmt, per_tok in ((W.KV_FP8, 132), (W.KV_FP4, 76), (W.KV_MXFP4, 68)):
        wl = W.build("b", [300, 517], [2, 3], topk=64, kv_format=fmt, seed=1)
        key_b, logit_b, small_b, flops = bench.algorithmic_bytes(wl)
        lmax = [max(wl.context_lens[:2]).item(), max(wl.context_lens[2:]).item()]
        assert key_b == per_tok * sum(lmax)
        assert flops == 2 * 64 * 128 * int(wl.context_lens.sum())
        elt = 4 if wl.logits_dtype == W.LOGITS_F32 else 2
        assert logit_b == elt * int(wl.context_lens.sum())
