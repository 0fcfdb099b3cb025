"""The seeded input generator: determinism, prefix property, workload shapes."""

import numpy as np
import torch

from mxfp4_activation_quant_gb300 import synth


def test_splitmix64_reference_values():
    # splitmix64 with state 0: the first outputs of the published generator
    # (state += golden gamma, then the finaliser) are the mix of k * gamma.
    w = synth.words(np.uint64(0), 0, 3)
    assert [int(v) for v in w] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_prefix():
    w = synth.WORKLOADS["prefill"]
    a = synth.make_inputs(w, M=6)
    b = synth.make_inputs(w, M=3)
    for k in a:
        if a[k].dim() == 2:
            assert torch.equal(a[k][:3], b[k])
        else:
            assert torch.equal(a[k], b[k])


def test_workload_shapes_and_distributions():
    d = synth.make_inputs(synth.WORKLOADS["decode"])
    assert d["x"].shape == (64, 7168) and d["x"].dtype == torch.bfloat16
    ch = synth.outlier_channels(1, 7168)
    assert len(ch) == 72
    x = d["x"].float()
    inner = np.setdiff1d(np.arange(7168), ch)
    assert 15 < x[:, ch].std().item() < 25 and 0.9 < x[:, inner].std().item() < 1.1
    assert 1.8 < d["residual"].float().std().item() < 2.2
    q = synth.make_inputs(synth.WORKLOADS["qknorm"], M=64)
    assert q["q_a"].shape == (64, 1536) and q["kv_a"].shape == (64, 512)
    assert 1.3 < q["kv_a"].float().std().item() < 1.5
    t = synth.make_inputs(synth.WORKLOADS["mxfp4"], M=16)["x"].float()
    assert t.abs().max().item() > 8           # heavy tail


def test_mxfp4_weights_are_seeded_and_in_range():
    q1, s1 = synth.mxfp4_weights(7, 40, 256)
    q2, s2 = synth.mxfp4_weights(7, 40, 256)
    assert q1.shape == (40, 128) and s1.shape == (40, 8)
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
    assert not torch.equal(q1, synth.mxfp4_weights(8, 40, 256)[0])
    s = s1.numpy()
    assert s.min() >= 118 and s.max() < 122
    nib = np.concatenate([(q1.numpy() & 0xF).ravel(), (q1.numpy() >> 4).ravel()])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.7 * nib.size / 16 and counts.max() < 1.3 * nib.size / 16
