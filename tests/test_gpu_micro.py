"""The special-function unit's exponential rate (sv_measure_ex2), the second
bound of the verify path: a plausible, repeatable figure on the device."""
import pytest
import torch

import speculative_decoding_verification_71_gb300 as svp

pytestmark = pytest.mark.gpu


def test_ex2_rate_is_plausible_and_repeatable():
    torch.cuda.set_device(0)
    a_clk, a_s = svp.measure_ex2(1024)
    b_clk, b_s = svp.measure_ex2(1024)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # an SM issues at most 128 lane operations per clock; a special-function
    # unit delivers a few to a few tens of exponentials per SM per clock
    assert 2.0 <= a_clk <= 128.0, a_clk
    assert abs(a_clk - b_clk) <= 0.05 * a_clk
    # per second: the per-clock rate times the SMs at a clock between 0.5 and 3 GHz
    assert a_clk * sms * 0.5e9 <= a_s <= a_clk * sms * 3.0e9, (a_clk, a_s)
