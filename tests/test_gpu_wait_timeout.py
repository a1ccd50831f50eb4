"""The bounded device wait, made to run out on purpose.

Every pipeline wait of the step's kernels is an mbarrier wait that gives up
after a fixed number of SM cycles and records kDevWaitTimeout (3) in the
engine's error word, so that a protocol slip ends a kernel instead of
hanging the device.  cbd_engine_test_wait_timeout runs that same wait, with
a short limit, in a one-warp kernel on a barrier that nothing completes (no
copy in flight, no tensor memory, no peer CTA).  The test checks that the
kernel returns, that cbd_engine_check reports CBD_EDEVICE with code 3 and
clears it, and that the next step of the tiny workload still matches the
oracle (logits max-abs <= 1e-2 * max|z|, mean-abs <= 2e-3)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import continuous_batching_decode_gb300 as cbd
    from oracle import model as om
    from tests import gpu_util as gu
    from tests.test_gpu_step import tiny_setup


def test_wait_runs_out_and_engine_recovers():
    from continuous_batching_decode_gb300 import build
    build.build()
    m = gu.Model("tiny", max_rows=512, max_slots=8, mbps=16)
    try:
        wl, pool, tables, nbps, rows, sampling = tiny_setup(m, 1)
        cbd.engine_check(m.e)
        with pytest.raises(cbd.CbdError):
            cbd.engine_test_wait_timeout(m.e, 0)           # limit out of range: refused on the host
        cbd.engine_test_wait_timeout(m.e, 1 << 20)
        torch.cuda.synchronize()                           # the kernel has returned
        with pytest.raises(cbd.CbdError) as ei:
            cbd.engine_check(m.e)
        assert ei.value.status == cbd.EDEVICE and "code 3" in str(ei.value)
        cbd.engine_check(m.e)                              # the word was cleared
        toks, z_gpu = gu.run_step(m, pool, rows, tables, nbps, sampling)
        om_ = m.oracle()
        prior = {s: c for s, c in enumerate(wl["contexts"])}
        kv = gu.oracle_kv_from_gpu(m, pool, tables, prior)
        kv[4] = om.SequenceKV(om_.cfg, 64)
        z = om.step(om_, kv, [(r[0], r[1], r[2], r[4]) for r in rows])
        gu.assert_logits_close(z_gpu, z, "step after a timed-out wait")
        pool.close()
    finally:
        m.close()
