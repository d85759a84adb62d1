"""Shared helpers of the parity tests: tolerances, comparisons, uploads."""
import numpy as np

from bit_affine_quantized_mlx_gb300 import synth

# Output tolerance for floating-point results, per output tensor:
#   max|y - y_ref| <= 1e-2 * max|y_ref|  and  ||y - y_ref||_2 / ||y_ref||_2 <= 5e-3.
MAX_ABS_REL = 1e-2
REL_L2 = 5e-3


def bf16_bits_to_f64(t):
    a = t.detach().cpu().numpy() if hasattr(t, "detach") else np.asarray(t)
    return synth.bf16_to_f32(a.view(np.uint16)).astype(np.float64)


def assert_close(got, want, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    err = np.abs(got - want).max()
    scale = np.abs(want).max()
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300)
    assert err <= MAX_ABS_REL * scale, f"{what}: max|err| {err:.3e} > 1e-2 * {scale:.3e}"
    assert rel <= REL_L2, f"{what}: rel L2 {rel:.3e} > 5e-3"
    return err / max(scale, 1e-300), rel


def assert_topk_equal(got_idx, got_w, ref, what=""):
    """Selected sets must be identical per token; weights compared per expert id.
    The order inside the top-k is a valid descending order of the GPU's fp32 logits; two
    selected logits closer than fp32 rounding may legitimately swap, so the set is compared."""
    gi = np.asarray(got_idx)
    ri = ref["idx"]
    for t in range(ri.shape[0]):
        assert sorted(gi[t].tolist()) == sorted(ri[t].tolist()), f"{what}: token {t} {gi[t]} vs {ri[t]}"
        assert len(set(gi[t].tolist())) == len(gi[t])
        if got_w is not None:
            gw = dict(zip(gi[t].tolist(), np.asarray(got_w)[t].tolist()))
            for e, p in zip(ri[t].tolist(), ref["p"][t].tolist()):
                assert abs(gw[e] - p) <= 1e-5, f"{what}: token {t} expert {e} p {gw[e]} vs {p}"
            # descending order of the reference logits up to fp32-level ties
            lg = ref["logits"][t][gi[t]]
            assert np.all(np.diff(lg) <= 1e-5)
