"""Forward + backward over batches that live in pinned host memory.

Plumbing around the C entry points: host<->device copies on two copy streams,
the kernels on a compute stream, and CUDA events between them.  Two slots,
each with its own device inputs, outputs and workspace, keep two batches in
flight, so batch i's inputs travel to the device and batch i-1's results
travel back while batch i-1 (then i) computes.  The only orderings are each
batch's copy-in -> compute -> copy-out chain and the reuse of a slot two
batches later (its copy-in waits until the slot's previous compute has read
its inputs; its compute waits until the slot's previous results were copied
out).
"""
from __future__ import annotations

import os
from typing import Callable, Dict, Optional

import torch

from . import Buffers, Opts, default_opts, flamia_bwd, flamia_fwd


def gpu_local_cpus(device) -> Optional[set]:
    """CPUs of the NUMA node the GPU is attached to (from sysfs), or None.

    Pinned host buffers are placed on the node of the thread that allocates
    them; allocating them from these CPUs keeps host<->device copies off the
    link between CPU sockets."""
    try:
        prop = torch.cuda.get_device_properties(torch.device(device))
        bdf = f"{prop.pci_domain_id:04x}:{prop.pci_bus_id:02x}:{prop.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bdf}/numa_node") as f:
            node = int(f.read().strip())
        if node < 0:
            return None
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            return parse_cpulist(f.read()) or None
    except (OSError, ValueError, AttributeError, RuntimeError):
        return None


def parse_cpulist(spec: str) -> set:
    """CPU numbers of a Linux CPU list ("0-3,8,10-11")."""
    cpus = set()
    for part in spec.strip().split(","):
        if not part:
            continue
        lo, _, hi = part.partition("-")
        cpus.update(range(int(lo), int(hi or lo) + 1))
    return cpus


def bind_to_gpu_node(device) -> bool:
    """Restrict this process to the GPU's local CPUs (True if done)."""
    cpus = gpu_local_cpus(device)
    if not cpus or not hasattr(os, "sched_setaffinity"):
        return False
    try:
        os.sched_setaffinity(0, cpus)
        return True
    except OSError:
        return False


INPUTS = ("q", "k", "v", "do")
OUTPUTS = ("out", "lse", "dq", "dk", "dv")


class _Slot:
    def __init__(self, T, n_docs, Hq, Hkv, d, device, opts=None):
        self.buf = Buffers(T, n_docs, Hq, Hkv, d, device=device, opts=opts)
        self.q = torch.empty(T, Hq, d, dtype=torch.bfloat16, device=device)
        self.k = torch.empty(T, Hkv, d, dtype=torch.bfloat16, device=device)
        self.v = torch.empty(T, Hkv, d, dtype=torch.bfloat16, device=device)
        self.do = torch.empty(T, Hq, d, dtype=torch.bfloat16, device=device)
        self.cu = torch.empty(n_docs + 1, dtype=torch.int32, device=device)
        self.copied_in = torch.cuda.Event()
        self.computed = torch.cuda.Event()
        self.copied_out = torch.cuda.Event()
        self.used = False


class HostPipeline:
    """Runs flamia_fwd + flamia_bwd on host batches with the copies overlapped.

    ``submit(host_in, host_out)`` enqueues one batch and returns at once.
    ``host_in`` maps q, k, v, do (bf16, [T,H,d]) and cu (int32, n_docs + 1) to
    pinned CPU tensors; ``host_out`` maps out, lse, dq, dk, dv to pinned CPU
    tensors of the shapes flamia_fwd / flamia_bwd write.  The host tensors of a
    batch must stay untouched until ``synchronize()`` (or until the batch two
    submissions later has been submitted and synchronized).  ``pre_step``, if
    given, runs on the compute stream before each batch's kernels.
    """

    def __init__(self, T: int, n_docs: int, Hq: int, Hkv: int, d: int, device="cuda",
                 opts: Optional[Opts] = None, pre_step: Optional[Callable[[], None]] = None):
        self.device = torch.device(device)
        self.opts = opts if opts is not None else default_opts()
        self.pre_step = pre_step
        self.slots = [_Slot(T, n_docs, Hq, Hkv, d, self.device, self.opts) for _ in range(2)]
        self.s_in = torch.cuda.Stream(self.device)
        self.s_compute = torch.cuda.Stream(self.device)
        self.s_out = torch.cuda.Stream(self.device)
        self.n = 0

    @property
    def copy_in_stream(self) -> torch.cuda.Stream:
        return self.s_in

    @property
    def copy_out_stream(self) -> torch.cuda.Stream:
        return self.s_out

    def submit(self, host_in: Dict[str, torch.Tensor], host_out: Dict[str, torch.Tensor]) -> None:
        s = self.slots[self.n % 2]
        with torch.cuda.stream(self.s_in):
            if s.used:
                self.s_in.wait_event(s.computed)
            for name in INPUTS:
                getattr(s, name).copy_(host_in[name], non_blocking=True)
            cu = host_in["cu"]
            if cu.numel() > s.cu.numel():
                raise ValueError("more documents than the pipeline was sized for")
            s.cu_n = cu.numel()
            s.cu[:cu.numel()].copy_(cu, non_blocking=True)
            s.copied_in.record(self.s_in)
        with torch.cuda.stream(self.s_compute):
            self.s_compute.wait_event(s.copied_in)
            if s.used:
                self.s_compute.wait_event(s.copied_out)
            if self.pre_step is not None:
                self.pre_step()
            B, cu_d = s.buf, s.cu[:s.cu_n]
            flamia_fwd(s.q, s.k, s.v, cu_d, B.out, B.lse, B.saved, B.work, self.opts, stream=self.s_compute)
            flamia_bwd(B.out, B.lse, s.do, cu_d, B.saved, B.dq, B.dk, B.dv, B.work, self.opts,
                       stream=self.s_compute)
            s.computed.record(self.s_compute)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(s.computed)
            for name in OUTPUTS:
                host_out[name].copy_(getattr(s.buf, name), non_blocking=True)
            s.copied_out.record(self.s_out)
        s.used = True
        self.n += 1

    def synchronize(self) -> None:
        for st in (self.s_in, self.s_compute, self.s_out):
            st.synchronize()

    @staticmethod
    def bytes_per_batch(host_in: Dict[str, torch.Tensor], host_out: Dict[str, torch.Tensor]):
        """(host->device, device->host) bytes one submission copies."""
        h2d = sum(host_in[n].numel() * host_in[n].element_size() for n in INPUTS + ("cu",))
        d2h = sum(host_out[n].numel() * host_out[n].element_size() for n in OUTPUTS)
        return h2d, d2h
