"""Failure detection on the GPU without a fault: every wait inside the decode kernel is
bounded, and a wait that runs out is reported to the host as KVARN_ETIMEOUT while the
CUDA context stays usable.

KVARN_FLAG_TEST_STALL makes one thread of the decode launch wait, before any copy is
issued, on a shared-memory word that nothing sets (include/kvarn.h). The pages have no
counterpart; this checks the library's own error path.
"""
import time

import numpy as np
import pytest

from quantized_kv_cache_seal_gb300 import kvarn as K
from quantized_kv_cache_seal_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _fill(cache, n=700):
    src = workloads.TokenSource(61, 0, 2)
    k, v = src.tokens(0, n)
    cache.append(0, [0], [n], torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())


def test_bounded_wait_reports_timeout_and_context_stays_usable():
    from quantized_kv_cache_seal_gb300.cache import KVarNCache
    stalled = KVarNCache(num_layers=1, max_seqs=1, num_q_heads=8, num_kv_heads=2, max_seq_len=2048,
                         flags=K.KVARN_FLAG_TEST_STALL)
    normal = KVarNCache(num_layers=1, max_seqs=1, num_q_heads=8, num_kv_heads=2, max_seq_len=2048)
    for c in (stalled, normal):
        _fill(c)
    q = torch.from_numpy(workloads.queries(62, 0, 1, 8)).cuda()
    torch.cuda.synchronize()
    t0 = time.time()
    out_s = stalled.decode_attention(0, [0], q)
    torch.cuda.synchronize()
    waited = time.time() - t0
    assert stalled.check_device_error() == 6  # KVARN_ETIMEOUT
    assert waited >= 1.0, waited              # the wait ran its limit, then gave up
    # the context is still usable, and the stalled launch finished its work
    out_n = normal.decode_attention(0, [0], q)
    assert normal.check_device_error() == 0
    assert torch.equal(out_s, out_n)
    # the check cleared the error word; a call on the normal cache right after is clean
    assert stalled.check_device_error() == 0
    out_again = normal.decode_attention(0, [0], q)
    assert torch.equal(out_again, out_n)
    assert np.isfinite(out_n.float().cpu().numpy()).all()
