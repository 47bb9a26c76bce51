"""Work hand-out of the attention kernels (FLAMIA Section 3.6.2).

The work list is sorted longest-first on the device; the persistent CTAs
either claim items at run time from a counter in the workspace (the default)
or walk the list in a fixed snake order.  Which CTA computes an item must not
change its result: O, LSE, dK, dV and dQ are compared bitwise between the
two (dQ with the order-independent fixed-point accumulation, since the
default fp32 reduce-adds arrive in a run-dependent order).

On workloads with more items than CTAs, every CTA's last claim fails and
every successful claim beyond the first round bumps the counter once, so the
counter ends at the number of items: that shows the dynamic claims ran.
"""
import numpy as np
import pytest
import torch

import precision_causal_attention_gb300 as F
import workloads as W
from tests.gpu_common import rel_fro

pytestmark = pytest.mark.gpu


def _skewed(d, seed):
    # one long document and many short ones: the shape that stresses scheduling
    rng = np.random.default_rng(seed)
    lens = [3000]
    while sum(lens) < 8192:
        lens.append(int(min(rng.integers(64, 513), 8192 - sum(lens))))
    return W.custom(lens, Hq=16, Hkv=4, d=d, seed=seed, T=8192)


def _run(w, schedule, exact=False, deterministic_dq=True):
    dev = torch.device("cuda:0")
    q, k, v, do = (w.tensors[n].to(dev) for n in ("q", "k", "v", "do"))
    cu = torch.from_numpy(np.asarray(w.cu_seqlens, np.int32)).to(dev)
    opts = F.default_opts(schedule=schedule, exact=exact, deterministic_dq=deterministic_dq)
    B = F.Buffers(w.T, w.n_docs, w.Hq, w.Hkv, w.d, opts=opts)
    F.flamia_fwd(q, k, v, cu, B.out, B.lse, B.saved, B.work, opts)
    torch.cuda.synchronize()
    fwd_claims = int(B.work[24:28].view(torch.int32).item())
    F.flamia_bwd(B.out, B.lse, do, cu, B.saved, B.dq, B.dk, B.dv, B.work, opts)
    torch.cuda.synchronize()
    bwd_claims = int(B.work[24:28].view(torch.int32).item())
    assert F.flamia_get_status() == 0
    return B, fwd_claims, bwd_claims


def _items(w, causal=True):
    lens = np.diff(np.asarray(w.cu_seqlens, np.int64))
    nt = (lens + 127) // 128
    per_head = int(nt.sum())
    return per_head * w.Hq, per_head * w.Hkv


@pytest.mark.parametrize("d,exact", [(64, False), (128, False), (64, True)], ids=["d64", "d128", "d64_exact"])
def test_dynamic_and_static_hand_out_agree_bitwise(d, exact):
    w = _skewed(d, seed=40 + d)
    dyn, fc, bc = _run(w, "dynamic", exact)
    sta, fc_s, bc_s = _run(w, "static", exact)
    n_fwd, n_bwd = _items(w)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    fwd_grid = sms * (2 if d == 64 else 1)
    # dynamic: the counter ends at the item count when the list is longer than the grid
    if n_fwd > fwd_grid:
        assert fc == n_fwd, (fc, n_fwd)
    if n_bwd > sms:
        assert bc == n_bwd, (bc, n_bwd)
    # static: nothing claims, the plan job's zero stays
    assert fc_s == 0 and bc_s == 0
    for key in ("out", "lse", "dk", "dv", "dq"):
        assert torch.equal(getattr(dyn, key), getattr(sta, key)), key
    # the default fp32 dQ agrees with the fixed-point one up to rounding
    fp, _, _ = _run(w, "dynamic", exact, deterministic_dq=False)
    assert rel_fro(fp.dq.float().cpu().numpy(), dyn.dq.float().cpu().numpy()) < 1e-3
