"""The seeded input generators: determinism, shapes, and the BF16 rounding they use."""
import numpy as np
import torch

from deterministic_top_key_gb300 import inputs


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, -2.5, 3.0039062, 1e-30, -1e30], np.float32)])
    ours = inputs.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = inputs.bf16_bits_to_f32(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_draw_is_deterministic_and_shaped():
    a = inputs.make("tiny")
    b = inputs.make("tiny")
    np.testing.assert_array_equal(a.q_bits, b.q_bits)
    np.testing.assert_array_equal(a.k_bits, b.k_bits)
    np.testing.assert_array_equal(a.w, b.w)
    assert a.q_bits.shape == (512, 64, 128) and a.k_bits.shape == (512, 128) and a.w.shape == (512, 64)
    assert a.top_k == 128 and a.num_segments == 1
    assert np.all(np.abs(a.w) <= 1.0)


def test_integer_variant_values():
    a = inputs.make("tiny", kind="int")
    q = inputs.bf16_bits_to_f32(a.q_bits)
    assert set(np.unique(q).tolist()) == {-2.0, -1.0, 0.0, 1.0, 2.0}
    assert set(np.unique(a.w).tolist()) <= {-1.0, 0.5, 1.0, 2.0}


def test_config_layouts():
    c = inputs.config("Z2")
    assert c["T"] == 16384 and c["Tkv"] == 270336
    cu_q, cu_k = np.asarray(c["cu_seqlens_q"]), np.asarray(c["cu_seqlens_k"])
    assert len(cu_q) == 17 and np.all(np.diff(cu_q) == 1024)
    assert np.array_equal(np.diff(cu_k), np.array([1024, 32768] * 8))
    c1 = inputs.config("C1")
    assert c1["q_causal_offsets"] == [61440] and c1["Tkv"] - c1["T"] == 61440


def test_z3_and_split_tail_layouts():
    """Z3cp totals as printed in the pages' table; every document splits into 32 chunks;
    the split-tail rows are the last 4 queries of one document."""
    c = inputs.config("Z3")
    assert c["T"] == 10624 and c["Tkv"] == 175296
    cu_q, cu_k = np.asarray(c["cu_seqlens_q"]), np.asarray(c["cu_seqlens_k"])
    assert len(cu_q) == 17
    tq, tk = np.diff(cu_q), np.diff(cu_k)
    docs = np.asarray(inputs.Z3_DOCS)
    assert np.array_equal(tq, np.repeat(docs // 32, 2))
    assert np.array_equal(tk[0::2], docs // 32) and np.array_equal(tk[1::2], docs)
    assert 4096 <= docs.min() and docs.max() <= 65536
    for name, tkv in (("A1", 22018), ("A2", 30466), ("A3", 41986)):
        a = inputs.config(name)
        assert a["T"] == 4 and a["Tkv"] == tkv and a["q_causal_offsets"] is None
