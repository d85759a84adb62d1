"""Host-side checks of the seeded input generator (no GPU)."""
import numpy as np
import torch

from bit_affine_quantized_mlx_gb300 import synth


def test_bf16_rounding_matches_torch():
    """Round-to-nearest-even to bf16 agrees with torch's CPU conversion (a library routine)."""
    rng = np.random.default_rng(0)
    f = np.concatenate([rng.normal(0, 1, 100000), rng.uniform(-1e-3, 1e-3, 1000),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 65504.0, 3.0e38])])
    f = f.astype(np.float32)
    mine = synth.bf16_from_f32(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)
    back = synth.bf16_to_f32(mine)
    assert np.array_equal(torch.from_numpy(back).numpy(),
                          torch.from_numpy(f).to(torch.bfloat16).float().numpy())


def test_draws_are_deterministic_and_keyed():
    a = synth.draw_q4(16, 128, 1, 2, 3)
    b = synth.draw_q4(16, 128, 1, 2, 3)
    c = synth.draw_q4(16, 128, 1, 2, 4)
    assert np.array_equal(a.w, b.w) and np.array_equal(a.s, b.s) and np.array_equal(a.b, b.b)
    assert not np.array_equal(a.w, c.w)
    x0 = synth.draw_x(256, (0, 0), 0, 0)
    assert np.array_equal(x0, synth.draw_x(256, (0, 0), 0, 0))
    assert not np.array_equal(x0, synth.draw_x(256, (0, 0), 0, 1))


def test_stack_expert_is_redrawable_alone():
    st = synth.draw_q4_stack(4, 32, 128, 5, 6)
    one = synth.draw_q4(32, 128, 5, 6, 2)
    assert np.array_equal(st.w[2], one.w) and np.array_equal(st.s[2], one.s)


def test_value_distributions():
    m = synth.draw_q4(512, 2048, 9, 9)
    s = synth.bf16_to_f32(m.s)
    b = synth.bf16_to_f32(m.b)
    assert s.min() >= 0.0019 and s.max() <= 0.0201
    ratio = b / s
    assert abs(ratio.mean() + 8.0) < 0.01 and abs(ratio.std() - 0.4) < 0.02
    q = (m.w[..., None] >> (np.arange(8, dtype=np.uint32) * 4)) & 0xF
    hist = np.bincount(q.ravel(), minlength=16) / q.size
    assert np.all(np.abs(hist - 1 / 16) < 0.002)


def test_workload_shapes():
    w = synth.WORKLOADS
    assert (w[1].H, w[1].E, w[1].k, w[1].I, w[1].shared, w[1].layers) == (2048, 256, 8, 512, True, 40)
    assert (w[4].E, w[4].k, w[4].layers) == (512, 10, 48)
    assert w[2].V == 151936 and w[3].tokens == (2048,) and w[3].router_bias
    L = w[0].layer(0)
    assert L.gate.w.shape == (16, 128, 32) and L.down.w.shape == (16, 256, 16)
    assert L.router.shape == (16, 256) and not L.has_shared
    # one routed expert at the decode shapes is 1,769,472 bytes
    e = synth.draw_q4(512, 2048, 0).nbytes * 2 + synth.draw_q4(2048, 512, 0).nbytes
    assert e == 1769472
