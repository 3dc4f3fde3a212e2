"""The seeded input generator: SplitMix64's published outputs, the value
distribution, heavy-tail rate and padding (CPU); CPU/GPU bit equality (GPU)."""
import numpy as np
import pytest

import synth


def test_splitmix64_published_outputs():
    # First outputs of SplitMix64 seeded with 0 (Steele, Lea and Flood 2014;
    # the reference implementation's well-known sequence).
    assert synth.splitmix64_outputs(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                              0x06C45D188009454F]


def test_values_distribution_and_padding():
    v = synth.values(7, synth.GRAD, 1, 0, 0, 400_000, 1e-3, 399_990)
    assert v.dtype == np.float32
    assert not v[399_990:].any()
    x = v[:399_990].astype(np.float64)
    assert abs(x.mean()) < 1e-5 and abs(x.std() / 1e-3 - 1) < 0.01
    assert np.abs(x).max() <= 1e-3 * np.sqrt(24) * (1 + 1e-6)


def test_heavy_tail_rate_and_bf16():
    f = synth.values(9, synth.GRAD, 2, 3, 0, 500_000, 1e-3, 500_000, heavy_tail=True)
    assert abs(np.mean(np.abs(f) > 5e-3) - 0.01) < 0.002
    b = synth.values(9, synth.GRAD, 2, 3, 0, 500_000, 1e-3, 500_000, heavy_tail=True,
                     dtype=synth.DTYPE_BF16)
    assert b.dtype == np.uint16
    back = (b.astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.abs(back - f) <= np.abs(f) * 2 ** -8)


def test_windows_agree_with_whole_stream():
    whole = synth.values(3, synth.MASTER, 0, 0, 0, 10_000, 0.02, 9_000)
    part = synth.values(3, synth.MASTER, 0, 0, 4_321, 9_999, 0.02, 9_000)
    assert np.array_equal(whole[4_321:9_999], part)


def test_keys_differ_by_rank_step_stream():
    ks = {synth.key(1, s, t, r) for s in range(3) for t in range(3) for r in range(8)}
    assert len(ks) == 72


@pytest.mark.gpu
def test_gpu_generator_matches_cpu(cuda):
    import torch
    for dt, tdt in [(synth.DTYPE_F32, torch.float32), (synth.DTYPE_BF16, torch.bfloat16)]:
        t = torch.empty(300_001, dtype=tdt, device=cuda)
        synth.fill_tensor(t, 11, synth.GRAD, 4, 5, 1_000_003, 1e-3, 1_250_000, heavy_tail=True)
        torch.cuda.synchronize()
        cpu = synth.values(11, synth.GRAD, 4, 5, 1_000_003, 1_300_004, 1e-3, 1_250_000,
                           heavy_tail=True, dtype=dt)
        got = t.cpu()
        got = got.numpy() if tdt == torch.float32 else got.view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, cpu)
