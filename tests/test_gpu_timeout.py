"""The bounded-wait timeout path, exercised without a fault or a hang.

trsm_set_wait_limit(0) makes the first wait of every item of the batched f32
small kernel (the one that streams systems through the TMA engine) expire at
once.  The kernel must then record TRSM_ERR_DEVICE_TIMEOUT (901) in the
device status word, let its copies in flight land (those waits keep the full
limit), leave B untouched and return; the context stays usable, and the same
solve with the limit restored matches the oracle."""
import numpy as np
import pytest

import trsm_inputs as ti
from gpu_util import assert_parity, gpu_solve_buffers, logical, oracle_buffers, storage_pair

pytestmark = pytest.mark.gpu
TIMEOUT = 901


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch

    import triangular_solve_gb300 as tg
    from triangular_solve_gb300 import build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    tg.load_library()
    return dict(torch=torch, tg=tg, oracle=oracle_mod)


@pytest.mark.parametrize("m", [64, 32])
def test_expired_wait_is_reported_and_the_context_stays_usable(env, m):
    torch, tg = env["torch"], env["tg"]
    n, batch = 64, 1024  # enough items (system x 64-column slice) for the persistent TMA kernel
    L, B = ti.generate("f32", m, n, batch, kind="dd64", seed=m)
    a, b, geo = storage_pair(L, B)
    assert tg.trsm_device_status(True) in (0, TIMEOUT)  # start from a clear word
    tg.trsm_set_wait_limit(0)
    try:
        raw = gpu_solve_buffers("f32", a, b, geo, 1.0, torch, tg)
    finally:
        tg.trsm_set_wait_limit(-1)
    assert tg.trsm_device_status(True) == TIMEOUT
    same = (raw == b) | (np.isnan(raw) & np.isnan(b))
    assert np.all(same), "an item was written although its copies were abandoned"
    assert tg.trsm_device_status(True) == 0  # cleared by the read above

    raw = gpu_solve_buffers("f32", a, b, geo, 1.0, torch, tg)
    ref = oracle_buffers("f32", a, b, geo, 1.0, env["oracle"])
    assert tg.trsm_device_status(True) == 0
    assert_parity("f32", logical(raw, geo), logical(ref, geo), f"after the timeout, m={m}")
