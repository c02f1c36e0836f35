"""The tensor-core instruction ceiling diagnostic (nvfp4_mma_ceiling): it runs for
every kind, and the block-scaled FP4 instruction (K = 64) takes the same clock
cycles as the BF16 one (K = 16), i.e. four times its rate per cycle."""

import pytest

import nvfp4_block_scaled_gb300 as nv

pytestmark = pytest.mark.gpu


def test_ceiling_kinds_and_ratio():
    bf = nv.mma_ceiling("bf16", 2048)
    f8 = nv.mma_ceiling("fp8", 2048)
    f4 = nv.mma_ceiling("nvf4", 2048)
    assert nv.device_error() == 0
    for tf, cyc in (bf, f8, f4):
        assert tf > 100.0 and cyc > 0.0
    assert 3.0 < f4[0] / bf[0] < 8.0
    assert 1.5 < f8[0] / bf[0] < 4.0


def test_ceiling_rejects_bad_arguments():
    with pytest.raises(nv.NVFP4Error) as e:
        nv.mma_ceiling("nvf4", 6)
    assert e.value.status == -1
