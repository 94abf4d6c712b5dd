"""Host-buffer drivers: run the forward on tensors that live in pinned host
memory.

``add_rmsnorm_fwd_host`` (the fast path on Grace-Blackwell): the kernel
reads x, residual and weight from pinned host memory and writes out and
residual_out back to it directly over the host link (zero copy); no device
buffers, no copies.  The C library sees host pointers and uses its
register-load variant, so the results are the same bits as a device call.

``HostPipeline`` (copy engines): the rows are cut into chunks and each chunk
is copied to the device, processed and copied back, with the copies
overlapped with the kernels.

The rows are cut into chunks.  Chunk c is copied host-to-device on one
stream, processed by the library's kernel on a second stream once its copy
is done, and copied back device-to-host on a third stream once its kernel is
done; so the upload of chunk c+1, the kernel of chunk c and the download of
chunk c-1 run at the same time (the host link carries both directions at
once).  Every row is computed by the same kernel as a single device call
would use, so the results are identical bit for bit.

The device staging buffers are allocated once per driver (through torch's
caching allocator) and reused.
"""
from __future__ import annotations

import torch

from . import DraddError, add_rmsnorm_fwd, add_rmsnorm_quant_fwd, lib


def _pinned_ptr(t, name: str, numel: int, dtypes) -> int:
    if t.device.type != "cpu" or not t.is_pinned():
        raise ValueError(f"{name} must be a pinned host tensor")
    if t.dtype not in dtypes or not t.is_contiguous() or t.numel() != numel:
        raise ValueError(f"{name}: expected a contiguous {dtypes[0]} tensor of {numel} elements")
    return t.data_ptr()


def add_rmsnorm_fwd_host(x_h, r_h, w_h, eps: float, outs_h, stream=None, quant: bool = False):
    """Residual-add + RMSNorm of pinned host tensors, read and written by the
    kernel directly over the host link.  x_h, r_h: [n_rows, hidden] bf16;
    w_h: [hidden] bf16; outs_h: (out, residual_out), or for quant
    (out_q int8, scale fp32 [n_rows], residual_out).  Enqueues on `stream`
    (default: the current stream of cuda:0 or the current device) and
    returns; synchronise the stream before reading the outputs."""
    import ctypes
    import torch
    bf16 = (torch.bfloat16, torch.int16)
    hidden = int(x_h.shape[-1])
    n_rows = x_h.numel() // hidden if hidden else 0
    n = n_rows * hidden
    if stream is None:
        stream = torch.cuda.current_stream()
    args_in = (_pinned_ptr(x_h, "x", n, bf16), _pinned_ptr(r_h, "residual", n, bf16),
               _pinned_ptr(w_h, "weight", hidden, bf16), ctypes.c_float(eps), n_rows, hidden, stream.cuda_stream)
    if quant:
        q_h, s_h, ro_h = outs_h
        st = lib().add_rmsnorm_quant_fwd(_pinned_ptr(q_h, "out_q", n, (torch.int8,)),
                                         _pinned_ptr(s_h, "scale", n_rows, (torch.float32,)),
                                         _pinned_ptr(ro_h, "residual_out", n, bf16), *args_in)
        where = "add_rmsnorm_quant_fwd"
    else:
        out_h, ro_h = outs_h
        st = lib().add_rmsnorm_fwd(_pinned_ptr(out_h, "out", n, bf16), _pinned_ptr(ro_h, "residual_out", n, bf16),
                                   *args_in)
        where = "add_rmsnorm_fwd"
    if st != 0:
        raise DraddError(st, where)
    return outs_h


class HostPipeline:
    """Reusable driver for one shape: n_rows x hidden, chunks of chunk_rows."""

    def __init__(self, n_rows: int, hidden: int, device, chunk_rows: int = 1024, quant: bool = False):
        self.n_rows, self.hidden, self.quant = int(n_rows), int(hidden), bool(quant)
        self.device = torch.device(device)
        cr = max(1, min(int(chunk_rows), max(1, self.n_rows)))
        while (cr * self.hidden) % 16:  # every chunk starts 16-byte aligned (int8 rows too)
            cr += 1
        self.chunk_rows = cr
        bf16 = dict(dtype=torch.bfloat16, device=self.device)
        self.x = torch.empty(self.n_rows, self.hidden, **bf16)
        self.r = torch.empty(self.n_rows, self.hidden, **bf16)
        self.ro = torch.empty(self.n_rows, self.hidden, **bf16)
        self.w = torch.empty(self.hidden, **bf16)
        if self.quant:
            self.q = torch.empty(self.n_rows, self.hidden, dtype=torch.int8, device=self.device)
            self.scale = torch.empty(self.n_rows, dtype=torch.float32, device=self.device)
        else:
            self.out = torch.empty(self.n_rows, self.hidden, **bf16)
        self.s_up = torch.cuda.Stream(self.device)
        self.s_run = torch.cuda.Stream(self.device)
        self.s_down = torch.cuda.Stream(self.device)

    def __call__(self, x_h, r_h, w_h, eps: float, outs_h):
        """x_h, r_h: host [n_rows, hidden] bf16 (pinned for overlap); w_h:
        host [hidden].  outs_h: host tensors to fill: (out, residual_out) or,
        for the int8 variant, (out_q, scale, residual_out).  Returns after
        enqueueing; synchronise `self.s_down` (or the device) to read them."""
        n, cr = self.n_rows, self.chunk_rows
        cur = torch.cuda.current_stream(self.device)
        self.s_up.wait_stream(cur)
        with torch.cuda.stream(self.s_up):
            self.w.copy_(w_h, non_blocking=True)
        for lo in range(0, n, cr):
            hi = min(n, lo + cr)
            with torch.cuda.stream(self.s_up):
                self.x[lo:hi].copy_(x_h[lo:hi], non_blocking=True)
                self.r[lo:hi].copy_(r_h[lo:hi], non_blocking=True)
                up = torch.cuda.Event()
                up.record(self.s_up)
            self.s_run.wait_event(up)
            if self.quant:
                add_rmsnorm_quant_fwd(self.x[lo:hi], self.r[lo:hi], self.w, eps, out_q=self.q[lo:hi],
                                      scale=self.scale[lo:hi], residual_out=self.ro[lo:hi],
                                      stream=self.s_run)
            else:
                add_rmsnorm_fwd(self.x[lo:hi], self.r[lo:hi], self.w, eps, out=self.out[lo:hi],
                                residual_out=self.ro[lo:hi], stream=self.s_run)
            ran = torch.cuda.Event()
            ran.record(self.s_run)
            self.s_down.wait_event(ran)
            with torch.cuda.stream(self.s_down):
                if self.quant:
                    q_h, s_h, ro_h = outs_h
                    q_h[lo:hi].copy_(self.q[lo:hi], non_blocking=True)
                    s_h[lo:hi].copy_(self.scale[lo:hi], non_blocking=True)
                else:
                    out_h, ro_h = outs_h
                    out_h[lo:hi].copy_(self.out[lo:hi], non_blocking=True)
                ro_h[lo:hi].copy_(self.ro[lo:hi], non_blocking=True)
        cur.wait_stream(self.s_down)
        return outs_h
