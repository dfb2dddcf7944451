"""Failure detection without a GPU fault: a device-side wait that runs out
of time is reported as PFA_ERR_TIMEOUT after a synchronise, the kernel exits
cleanly (its copies and tensor-core work drained, tensor memory freed), and
the context stays usable for the next call."""
import pytest

import chunked_causal_gqa_gb300 as pkg
import oracle
from chunked_causal_gqa_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (512, "bf16"), (128, "f32")])
def test_forced_wait_timeout_is_reported_and_context_survives(D, dtype):
    q, k, v = W.make_random(100, 40, 8, 2, D, dtype, seed=51)
    d = G.dev()
    qd, kd, vd = q.to(d), k.to(d), v.to(d)
    pkg.debug_configure(wait_limit_ms=50.0, force_timeout=True)
    try:
        pkg.prefill_attention(qd, kd, vd)
        status = pkg.last_device_error()
    finally:
        pkg.debug_configure(0.0, False)
    assert status == -7, pkg.status_string(status)
    assert pkg.last_device_error() == 0          # the word was cleared
    got = G.to_np(G.run(q, k, v))                # the context still works
    G.check(got, oracle.prefill_attention(q, k, v), dtype, "after timeout")
