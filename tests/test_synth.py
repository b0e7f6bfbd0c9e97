"""The seeded input generator: bf16 rounding and reproducibility (CPU only)."""
import numpy as np
import torch

from top_sparse_attention_exact_gb300 import synth


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 50,
                        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40, np.inf, -np.inf], np.float32)])
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = synth.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_generator_shapes_and_determinism():
    w = synth.scaled(synth.WORKLOADS["qwen7b_16k"], L0=512, steps=8, seeds=(7,))
    a = synth.generate(w)
    b = synth.generate(w)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    k, v, qp, qd = a
    assert k.shape == (1, 4, 520, 128) and v.shape == k.shape
    assert qp.shape == (1, 28, 32, 128) and qd.shape == (8, 1, 28, 128)
    assert k.dtype == np.uint16


def test_generator_topic_structure():
    # consecutive queries of one head are mostly on the same topic: high cosine
    w = synth.scaled(synth.WORKLOADS["tiny_1h_2k"], L0=256, steps=64)
    _, _, _, qd = synth.generate(w)
    q = synth.bf16_bits_to_f32(qd[:, 0, 0]).astype(np.float64)
    qn = q / np.linalg.norm(q, axis=1, keepdims=True)
    cos = (qn[1:] * qn[:-1]).sum(1)
    assert (cos > 0.85).mean() > 0.6
