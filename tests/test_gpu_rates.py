"""The tensor-core rate measurement the bench uses for its prompt denominators: it runs through the C
ABI and returns rates of the right order for this GPU (dense fp16 on tcgen05 in the PFLOP/s range;
int8 on the warp-level mma.sync path, which is the only int8 tensor path on sm_103a)."""
import pytest

import sparse_selection_attention_gb300 as qsa

pytestmark = pytest.mark.gpu


def test_f16_and_int8_rates():
    f16 = qsa.measure_tc_rate(qsa.QSA_TC_KIND_F16, 3000)
    i8 = qsa.measure_tc_rate(qsa.QSA_TC_KIND_I8, 20)
    print(f"RATES f16 tcgen05 {f16 / 1e12:.1f} TFLOP/s, s8 mma.sync {i8 / 1e12:.1f} TOP/s")
    assert 2e14 < f16 < 5e15
    assert 1e13 < i8 < 5e15
    assert qsa.get_device_error() == 0
