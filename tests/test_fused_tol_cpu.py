"""CPU checks of the fused-projection tolerance (tests/_fused_tol.py): the
oracle's own results pass it, and results with a planted mistake (a scale one
fp16 step off in every group, a code off by one, a Q value off by an ulp) fail
it.  So the GPU tests that use it cannot pass vacuously."""
import numpy as np
import pytest

import oracle
from serving_tcgen05_streamed_gb300 import inputs
from tests._fused_tol import check_kv, check_q, head_bounds
from tests._util import bits16


@pytest.fixture(scope="module")
def h3_rows():
    # H3 width (56 heads, K = 7168), Q/K RMSNorm, 6 token rows
    x, w, qn, kn = inputs.block_inputs(inputs.MID, n=6)
    xb, wb = bits16(x), bits16(w)
    ref = oracle.qkv_proj(xb, wb, q_norm_w=qn.numpy(), k_norm_w=kn.numpy())
    return ref, head_bounds(xb, wb, qn.numpy(), kn.numpy())


def test_the_oracle_passes_its_own_tolerance(h3_rows):
    ref, b = h3_rows
    for n in ("k", "v"):
        c = check_kv(ref[f"{n}_codes"], ref[f"{n}_scales"], ref[f"{n}_codes"], ref[f"{n}_scales"], ref[f"{n}_rot"],
                     b[n], 4, 32, n)
        assert c["scales_differing"] == 0 and c["codes_differing"] == 0
    assert check_q(ref["q_bf16"], ref["q_f32"], ref["q_bf16"], b["q"])["q_differing"] == 0


def test_planted_mistakes_fail(h3_rows):
    ref, b = h3_rows
    up = ref["v_scales"] + 1  # every scale one fp16 step up
    with pytest.raises(AssertionError):
        check_kv(ref["v_codes"], up, ref["v_codes"], ref["v_scales"], ref["v_rot"], b["v"], 4, 32, "v")
    codes = ref["k_codes"].copy()
    codes[2, 7, 5] ^= 0x10  # one element's code changed
    with pytest.raises(AssertionError):
        check_kv(codes, ref["k_scales"], ref["k_codes"], ref["k_scales"], ref["k_rot"], b["k"], 4, 32, "k")
    q = ref["q_bf16"].copy()
    q[0, 100] += 2  # two BF16 ulps
    with pytest.raises(AssertionError):
        check_q(q, ref["q_f32"], ref["q_bf16"], b["q"])


def test_bounds_are_far_below_the_quantisation_step(h3_rows):
    # the y bound is a small fraction of a code step, so a differing code is
    # accepted only very close to a rounding boundary
    ref, b = h3_rows
    y = ref["v_rot"].reshape(6, 56, 4, 32).astype(np.float64)
    s = np.abs(y).max(-1) / 7
    assert np.median(2 * b["v"][:, :, None] / s) < 0.01
