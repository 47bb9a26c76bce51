"""The on-chip wait timeout, made to happen on purpose (no GPU fault involved).

Every mbarrier wait in the kernels is bounded in wall-clock time; a wait that
runs out records FLAMIA_STATUS_TIMEOUT in the device status word, and the
kernel winds down: the producer lets its in-flight copies land, the MMA
issuers wait for their tensor-core work, tensor memory is freed, and the CTA
exits.  flamia_debug_set_item_limit(1) makes every forward CTA stop handing
out work after its first item without sending the end-of-work marker, so the
waits for a next item are waits on a barrier nothing completes.  The test
checks that the call reports the timeout and that the next call on the same
context is clean and correct.
"""
import time

import numpy as np
import pytest

import precision_causal_attention_gb300 as F
import workloads as W
from oracle import blocks as OB
from oracle import simulated as OS
from tests.gpu_common import run_gpu, np_inputs, rel_fro

pytestmark = pytest.mark.gpu

FLAMIA_STATUS_TIMEOUT = 2


def test_forward_wait_timeout_is_reported_and_the_context_stays_usable():
    w = W.tiny()
    F.flamia_debug_set_item_limit(1)
    try:
        t0 = time.time()
        res = run_gpu(w, do_bwd=False)
        elapsed = time.time() - t0
    finally:
        F.flamia_debug_set_item_limit(0)
    assert res["status"] == FLAMIA_STATUS_TIMEOUT
    # the waits give up after their wall-clock budget (about 2 s), not later
    assert elapsed < 30.0, elapsed
    # the next calls on the same context: no status, and the oracle's results
    good = run_gpu(w)
    assert good["status"] == 0
    x = np_inputs(w)
    m = OB.in_doc_mask(w.cu_seqlens, w.T)
    f = OS.forward(x["q"], x["k"], x["v"], w.cu_seqlens)
    b = OS.backward(x["q"], x["k"], x["v"], f["O_bf16"], f["lse"], x["do"], w.cu_seqlens)
    assert rel_fro(good["out"][m], f["O"][m]) <= 1e-2
    for key in ("dq", "dk", "dv"):
        assert rel_fro(good[key][m], b[key][m]) <= 3e-2, key
