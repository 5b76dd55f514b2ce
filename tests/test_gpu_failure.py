"""The bounded waits' give-up path, made to run without a GPU fault.

Every pipeline wait of the expert-FFN kernels is bounded.  The test hook
qre_debug_wait_test lowers the bound to a few microseconds and delays one warp
of one CTA by 20 ms before it signals its first stage, so the
stage's issuer runs out of time: the kernel must record QRE_DEV_TIMEOUT, make
the CTA's other waits give up, let the tensor core finish what was issued, free
its tensor memory and return.  The same process then runs the layer again with
the default bound and must get the same bits as before and a clean status: a
CTA that had kept its tensor memory would leave the next kernel nothing to
allocate.  Nothing here traps, faults or waits without a bound.
"""

import numpy as np
import pytest

import synthetic
import quantized_routed_expert_03_gb300 as qre

from gpu_support import BuiltLayer, numpy_source
from test_gpu_layer import MID, ODD, _check_layer, _inputs, _run

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
LIMIT_NS = 5_000          # 5 us
STALL_NS = 20_000_000     # 20 ms


# H 512, I 512: both decode phases take the FP8 kernel (whole 128-element stages
# in every K slice); MID (I 256) and ODD (G 64) take the fp16-code kernel.
FP8 = synthetic.LayerConfig("fp8", 512, 512, 32, 4, 128, 8)


@pytest.mark.parametrize("cfg,T,tol", [(FP8, 1, 1e-5), (FP8, 8, 1e-5), (MID, 8, 1e-5), (ODD, 5, 1e-5),
                                       (MID, 40, 1e-3)],
                         ids=["fp8_decode_T1", "fp8_decode_T8", "fp16_decode_T8", "fp16_decode_G64", "prefill_T40"])
def test_wait_runs_out_then_next_call_is_clean(cfg, T, tol):
    built = BuiltLayer(cfg.hidden, cfg.inter, cfg.n_experts, cfg.top_k, cfg.group, T, DEV, numpy_source(cfg))
    x_bits, wr, _ = _inputs(cfg, T, step=21)
    qre.qre_clear_device_status()
    before = _run(built, x_bits, wr, None)
    assert qre.qre_read_device_status() == 0

    qre.qre_debug_wait_test(LIMIT_NS, STALL_NS)
    try:
        _run(built, x_bits, wr, None)                 # returns (the copy back synchronizes)
        status = qre.qre_read_device_status()
    finally:
        qre.qre_debug_wait_test(0, 0)
    assert status & qre.QRE_DEV_TIMEOUT, f"status {status:#x}"

    qre.qre_clear_device_status()
    for _ in range(2):
        after = _run(built, x_bits, wr, None)
        np.testing.assert_array_equal(after["expert_out"], before["expert_out"])
        np.testing.assert_array_equal(after["y"], before["y"])
    assert qre.qre_read_device_status() == 0
    _check_layer(built, after, built.oracle_layer(x_bits, wr, None), tol=tol)
