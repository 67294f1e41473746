"""Pins for the seeded input generator (synth/): published SplitMix64 outputs,
vectorised == scalar form, distribution shape and the routing counts."""
import numpy as np
import torch

import synth


def test_splitmix64_published_vectors():
    # SplitMix64 from state 0: the first three outputs as commonly published
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert synth.splitmix64_py(0, 3) == want
    got = [int(v) & (2 ** 64 - 1) for v in synth.splitmix64(0, 0, 3)]
    assert got == want


def test_vectorised_matches_scalar():
    for stream in (1, 8 * 5 + 2, 2 ** 40 + 3):
        py = synth.splitmix64_py(stream, 50)
        vec = [int(v) & (2 ** 64 - 1) for v in synth.splitmix64(stream, 0, 50)]
        assert py == vec
        tail = [int(v) & (2 ** 64 - 1) for v in synth.splitmix64(stream, 20, 30)]
        assert tail == py[20:]


def test_normals_and_outliers():
    z = synth.normal(0, 200001)
    assert abs(float(z.mean())) < 0.01 and abs(float(z.std()) - 1) < 0.01
    a = synth.activation(0, 64, 7168)
    assert a.dtype == torch.bfloat16
    ch = synth.outlier_channels(0, 7168)
    assert ch.numel() == 7 and len(set(ch.tolist())) == 7
    col_std = a.float().std(dim=0)
    assert float(col_std[ch].min()) > 10 and float(np.delete(col_std.numpy(), ch.numpy()).max()) < 2
    assert synth.outlier_channels(0, 768).numel() == 1
    w = synth.weight(0, 128, 256)
    assert abs(float(w.float().std()) - 0.02) < 0.002


def test_moe_routing_counts():
    c = synth.moe_routing(0, 4096, 128, 8)
    assert int(c.sum()) == 4096 * 8 and c.numel() == 128
    row = synth.moe_offsets(c)
    assert int(row[-1]) == 32768 and row.numel() == 129 and bool((row[1:] >= row[:-1]).all())
