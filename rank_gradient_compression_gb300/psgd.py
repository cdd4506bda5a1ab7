"""ctypes binding of libpsgd.so (psgd.h). It only marshals arguments.

Every step of the computation runs in the CUDA library. PyTorch supplies device
memory and the current stream. If the shared library is missing or fails to load,
importing the binding raises; there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, byref, c_double, c_int32, c_int64, c_size_t, c_uint32, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("PSGD_LIB", os.path.join(HERE, "libpsgd.so"))

PSGD_F32, PSGD_F16, PSGD_BF16 = 0, 1, 2
PSGD_OK, PSGD_EINVAL, PSGD_ECUDA, PSGD_EUNSUPPORTED, PSGD_ETIMEOUT = range(5)
PSGD_FLAG_SIMT, PSGD_FLAG_MASK, PSGD_FLAG_STOP_AFTER_INGEST = 0x1, 0x2, 0x4
PSGD_FLAG_DEBUG_EXPIRE_WAIT = 0x8
PSGD_FLAG_EXCHANGE = 0x10

DTYPE_CODE = {"f32": PSGD_F32, "f16": PSGD_F16, "bf16": PSGD_BF16}

# Symbols that psgd.h declares (checked by the CPU test suite).
EXPORTS = ("psgd_workspace_size", "psgd_mask_offset", "psgd_mask_words", "psgd_init",
           "psgd_step", "psgd_check", "psgd_finalize", "psgd_strerror", "psgd_last_error",
           "psgd_debug_m", "psgd_debug_phat", "psgd_engine", "psgd_profile_begin",
           "psgd_profile_end", "psgd_launch_count", "psgd_debug_orth",
           "psgd_orthonormalize_static", "psgd_scale_update", "psgd_clip_adam_workspace_size",
           "psgd_clip_adam", "psgd_reduce_uncompressed", "psgd_step_p", "psgd_step_q",
           "psgd_step_e", "psgd_exchange_p", "psgd_exchange_q", "psgd_exchange_counts")
PSGD_STATIC_MAX_ROWS, PSGD_STATIC_MAX_COLS = 16384, 128
PSGD_MAX_ORTH_PASSES = 4
PSGD_ADAM_MAX_TENSORS = 512
PSGD_UNC_MAX_WORKERS = 16
PSGD_NUM_PHASES = 7
PHASES = ("ingest", "skip_unc", "pgemm", "orth", "qgemm", "qreduce", "decomp")


class psgd_shape(ctypes.Structure):
    _fields_ = [("m", c_int64), ("n", c_int64)]


class psgd_config(ctypes.Structure):
    _fields_ = [("num_blocks", c_int32), ("mats_per_block", c_int32), ("num_workers", c_int32),
                ("rank", c_int32), ("shapes", POINTER(psgd_shape)), ("grad_dtype", c_int32),
                ("err_dtype", c_int32), ("unc_len", c_int64), ("skip_fraction", c_double),
                ("flags", c_uint32)]


class psgd_step_args(ctypes.Structure):
    _fields_ = [("grads", POINTER(c_void_p)), ("errs", POINTER(c_void_p)),
                ("q_state", POINTER(c_void_p)), ("scales", POINTER(ctypes.c_float)),
                ("ghat", POINTER(c_void_p)), ("unc_in", POINTER(c_void_p)),
                ("unc_out", POINTER(c_void_p)), ("counts", c_void_p), ("skip", c_void_p),
                ("mask_bits", c_void_p), ("scales_device", c_void_p)]


class psgd_adam_args(ctypes.Structure):
    _fields_ = [("num_tensors", c_int32), ("grads", POINTER(c_void_p)),
                ("params", POINTER(c_void_p)), ("exp_avg", POINTER(c_void_p)),
                ("exp_avg_sq", POINTER(c_void_p)), ("numel", POINTER(c_int64)),
                ("block", POINTER(c_int32)), ("skip", c_void_p), ("num_blocks", c_int32),
                ("max_norm", c_double), ("lr", c_double), ("beta1", c_double),
                ("beta2", c_double), ("eps", c_double), ("step", c_int32),
                ("norm_out", c_void_p)]


class PSGDError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"psgd status {status}: {msg}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libpsgd.so not built ({LIB_PATH}); run "
                          "`python -m rank_gradient_compression_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    lib.psgd_workspace_size.restype = c_size_t
    lib.psgd_workspace_size.argtypes = [POINTER(psgd_config)]
    lib.psgd_mask_offset.restype = c_int64
    lib.psgd_mask_offset.argtypes = [POINTER(psgd_config), c_int32, c_int32, c_int32]
    lib.psgd_mask_words.restype = c_int64
    lib.psgd_mask_words.argtypes = [POINTER(psgd_config)]
    lib.psgd_init.restype = c_int32
    lib.psgd_init.argtypes = [POINTER(psgd_config), c_void_p, c_size_t, c_void_p, POINTER(c_void_p)]
    lib.psgd_step.restype = c_int32
    lib.psgd_step.argtypes = [c_void_p, POINTER(psgd_step_args), c_void_p]
    for name in ("psgd_step_p",):
        getattr(lib, name).restype = c_int32
        getattr(lib, name).argtypes = [c_void_p, POINTER(psgd_step_args), c_void_p]
    lib.psgd_step_q.restype = c_int32
    lib.psgd_step_q.argtypes = [c_void_p, POINTER(psgd_step_args), c_void_p, c_int32, c_void_p]
    lib.psgd_step_e.restype = c_int32
    lib.psgd_step_e.argtypes = [c_void_p, POINTER(psgd_step_args), c_int32, c_void_p]
    for name in ("psgd_exchange_p", "psgd_exchange_q"):
        getattr(lib, name).restype = c_void_p
        getattr(lib, name).argtypes = [c_void_p, c_int32, c_int32]
    lib.psgd_exchange_counts.restype = c_void_p
    lib.psgd_exchange_counts.argtypes = [c_void_p]
    lib.psgd_check.restype = c_int32
    lib.psgd_check.argtypes = [c_void_p, c_void_p]
    lib.psgd_finalize.restype = c_int32
    lib.psgd_finalize.argtypes = [c_void_p]
    lib.psgd_strerror.restype = ctypes.c_char_p
    lib.psgd_strerror.argtypes = [c_int32]
    lib.psgd_last_error.restype = ctypes.c_char_p
    lib.psgd_last_error.argtypes = []
    lib.psgd_debug_m.restype = c_void_p
    lib.psgd_debug_m.argtypes = [c_void_p, c_int32, c_int32, c_int32]
    lib.psgd_debug_phat.restype = c_void_p
    lib.psgd_debug_phat.argtypes = [c_void_p, c_int32, c_int32]
    lib.psgd_engine.restype = ctypes.c_char_p
    lib.psgd_engine.argtypes = [c_void_p]
    lib.psgd_profile_begin.restype = c_int32
    lib.psgd_profile_begin.argtypes = [c_void_p, c_int32]
    lib.psgd_profile_end.restype = c_int32
    lib.psgd_profile_end.argtypes = [c_void_p, POINTER(c_double), POINTER(c_int32)]
    lib.psgd_launch_count.restype = c_int64
    lib.psgd_launch_count.argtypes = [c_void_p]
    lib.psgd_debug_orth.restype = c_int32
    lib.psgd_debug_orth.argtypes = [c_void_p, c_int32, c_int32, POINTER(c_int32), c_void_p]
    lib.psgd_orthonormalize_static.restype = c_int32
    lib.psgd_orthonormalize_static.argtypes = [c_void_p, c_void_p, c_int64, c_int32, c_void_p]
    lib.psgd_clip_adam_workspace_size.restype = c_size_t
    lib.psgd_clip_adam_workspace_size.argtypes = [c_int32, POINTER(c_int64)]
    lib.psgd_clip_adam.restype = c_int32
    lib.psgd_clip_adam.argtypes = [POINTER(psgd_adam_args), c_void_p, c_size_t, c_void_p]
    lib.psgd_reduce_uncompressed.restype = c_int32
    lib.psgd_reduce_uncompressed.argtypes = [c_int32, POINTER(c_void_p), c_int64, ctypes.c_float,
                                             c_void_p, c_void_p, c_void_p, c_void_p]
    lib.psgd_scale_update.restype = c_int32
    lib.psgd_scale_update.argtypes = [c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_double,
                                      c_double, c_int32, c_void_p]
    return lib


lib = _load()


def _check(status: int):
    if status != PSGD_OK:
        raise PSGDError(status, lib.psgd_last_error().decode(errors="replace"))


def make_config(shapes, blocks, workers, rank, dtype, unc_len=0, skip_fraction=1.0, flags=0):
    """psgd_config plus the shape array it points to (keep both alive together)."""
    arr = (psgd_shape * len(shapes))(*[psgd_shape(int(m), int(n)) for m, n in shapes])
    cfg = psgd_config(int(blocks), len(shapes), int(workers), int(rank),
                      ctypes.cast(arr, POINTER(psgd_shape)), DTYPE_CODE[dtype], DTYPE_CODE[dtype],
                      int(unc_len), float(skip_fraction), int(flags))
    return cfg, arr


# Same names as the C ABI -------------------------------------------------------------
def psgd_workspace_size(cfg) -> int:
    return int(lib.psgd_workspace_size(byref(cfg)))


def psgd_mask_words(cfg) -> int:
    return int(lib.psgd_mask_words(byref(cfg)))


def psgd_mask_offset(cfg, b, j, w) -> int:
    return int(lib.psgd_mask_offset(byref(cfg), b, j, w))


def psgd_init(cfg, workspace_ptr: int, ws_bytes: int, stream: int) -> int:
    h = c_void_p()
    _check(lib.psgd_init(byref(cfg), c_void_p(workspace_ptr), ws_bytes, c_void_p(stream), byref(h)))
    return h.value


def psgd_step(handle: int, args: psgd_step_args, stream: int):
    _check(lib.psgd_step(c_void_p(handle), byref(args), c_void_p(stream)))


def psgd_step_p(handle: int, args: psgd_step_args, stream: int):
    _check(lib.psgd_step_p(c_void_p(handle), byref(args), c_void_p(stream)))


def psgd_step_q(handle: int, args: psgd_step_args, block_counts_ptr: int, total_workers: int,
                stream: int):
    _check(lib.psgd_step_q(c_void_p(handle), byref(args), c_void_p(block_counts_ptr),
                           int(total_workers), c_void_p(stream)))


def psgd_step_e(handle: int, args: psgd_step_args, total_workers: int, stream: int):
    _check(lib.psgd_step_e(c_void_p(handle), byref(args), int(total_workers), c_void_p(stream)))


def psgd_exchange_p(handle: int, b: int, j: int) -> int:
    return lib.psgd_exchange_p(c_void_p(handle), b, j) or 0


def psgd_exchange_q(handle: int, b: int, j: int) -> int:
    return lib.psgd_exchange_q(c_void_p(handle), b, j) or 0


def psgd_exchange_counts(handle: int) -> int:
    return lib.psgd_exchange_counts(c_void_p(handle)) or 0


def psgd_check(handle: int, stream: int):
    _check(lib.psgd_check(c_void_p(handle), c_void_p(stream)))


def psgd_finalize(handle: int):
    _check(lib.psgd_finalize(c_void_p(handle)))


def psgd_strerror(status: int) -> str:
    return lib.psgd_strerror(status).decode()


def psgd_engine(handle: int) -> str:
    return lib.psgd_engine(c_void_p(handle)).decode()


def psgd_profile_begin(handle: int, max_steps: int):
    _check(lib.psgd_profile_begin(c_void_p(handle), int(max_steps)))


def psgd_profile_end(handle: int):
    """Returns ({phase: summed ms}, profiled steps)."""
    ms = (c_double * PSGD_NUM_PHASES)()
    steps = c_int32()
    _check(lib.psgd_profile_end(c_void_p(handle), ms, byref(steps)))
    return dict(zip(PHASES, list(ms))), steps.value


def psgd_launch_count(handle: int) -> int:
    return int(lib.psgd_launch_count(c_void_p(handle)))


def psgd_orthonormalize_static(p_ptr: int, phat_ptr: int, m: int, r: int, stream: int):
    """P^ <- orthonormal basis of span(P), P and P^ dense fp32 m x r on the device, with
    the library's fixed scratch array (no allocation, no handle)."""
    _check(lib.psgd_orthonormalize_static(c_void_p(p_ptr), c_void_p(phat_ptr), int(m), int(r),
                                          c_void_p(stream)))


def psgd_scale_update(num_blocks: int, num_workers: int, counts_ptr: int, scale_ptr: int,
                      streak_ptr: int, backoff: float, growth: float, interval: int,
                      stream: int):
    """Per-resblock dynamic scale update on the device, from a finished step's counts:
    scale[b] *= backoff when block b had a nonfinite entry, else *= growth after
    `interval` consecutive finite steps (streak[b] counts them)."""
    _check(lib.psgd_scale_update(int(num_blocks), int(num_workers), c_void_p(counts_ptr),
                                 c_void_p(scale_ptr), c_void_p(streak_ptr), float(backoff),
                                 float(growth), int(interval), c_void_p(stream)))


def psgd_clip_adam_workspace_size(numel) -> int:
    arr = (c_int64 * len(numel))(*[int(x) for x in numel])
    return int(lib.psgd_clip_adam_workspace_size(len(numel), arr))


def psgd_clip_adam(grads, params, exp_avg, exp_avg_sq, numel, workspace_ptr, ws_bytes, stream,
                   lr, beta1=0.9, beta2=0.999, eps=1e-8, step=1, max_norm=0.0, block=None,
                   skip_ptr=0, num_blocks=0, norm_out_ptr=0):
    """Global-norm clip + one Adam step on lists of device pointers (fp32 tensors)."""
    T = len(grads)
    p = lambda xs: (c_void_p * T)(*[int(x) for x in xs])
    args = psgd_adam_args(T, p(grads), p(params), p(exp_avg), p(exp_avg_sq),
                          (c_int64 * T)(*[int(x) for x in numel]),
                          (c_int32 * T)(*[int(x) for x in block]) if block is not None else None,
                          c_void_p(skip_ptr), int(num_blocks), float(max_norm), float(lr),
                          float(beta1), float(beta2), float(eps), int(step), c_void_p(norm_out_ptr))
    _check(lib.psgd_clip_adam(byref(args), c_void_p(workspace_ptr), int(ws_bytes), c_void_p(stream)))


def psgd_reduce_uncompressed(in_ptrs, length: int, scale: float, out_ptr: int, counts_ptr: int,
                             skip_ptr: int = 0, stream: int = 0):
    """out = mean over workers of the unscaled, nonfinite-zeroed fp32 inputs (device pointers)."""
    W = len(in_ptrs)
    arr = (c_void_p * max(W, 1))(*[int(x) for x in in_ptrs])
    _check(lib.psgd_reduce_uncompressed(W, arr, int(length), float(scale), c_void_p(out_ptr),
                                        c_void_p(counts_ptr), c_void_p(skip_ptr), c_void_p(stream)))


def _ptrs(tensors):
    return (c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])


class PowerSGD:
    """Owns one psgd handle, its workspace and its count/skip outputs (torch tensors).

    ``step`` takes nested lists of CUDA tensors, grads[b][j][w], errs[b][j][w],
    q[b][j], ghat[b][j], unc_in[b][w] and unc_out[b], plus host scales[b] or, with
    ``scales_device`` (a CUDA fp32 tensor of B scales), scales read on the device. It
    enqueues one psgd_step on the current torch stream.
    """

    def __init__(self, shapes, blocks, workers, rank, dtype, unc_len=0, skip_fraction=1.0,
                 flags=0, device=None):
        import torch
        self.torch = torch
        self.shapes = [tuple(int(x) for x in s) for s in shapes]
        self.B, self.J, self.W, self.r = int(blocks), len(shapes), int(workers), int(rank)
        self.unc_len, self.flags = int(unc_len), int(flags)
        self.device = torch.device(device or "cuda")
        self.cfg, self._shape_arr = make_config(self.shapes, blocks, workers, rank, dtype, unc_len,
                                                skip_fraction, flags)
        ws = psgd_workspace_size(self.cfg)
        if ws == 0:
            raise PSGDError(PSGD_EINVAL, lib.psgd_last_error().decode())
        self.workspace = torch.empty(ws + 256, dtype=torch.uint8, device=self.device)
        base = self.workspace.data_ptr()
        self._ws_ptr = (base + 255) // 256 * 256
        self.counts = torch.zeros(self.B * self.W, dtype=torch.int64, device=self.device)
        self.skip = torch.zeros(self.B, dtype=torch.uint8, device=self.device)
        self.mask = None
        if flags & PSGD_FLAG_MASK:
            self.mask = torch.zeros(psgd_mask_words(self.cfg), dtype=torch.int32, device=self.device)
        stream = torch.cuda.current_stream(self.device).cuda_stream
        self.handle = psgd_init(self.cfg, self._ws_ptr, ws, stream)
        self.engine = psgd_engine(self.handle)

    def _args(self, grads, errs, q, scales, ghat, unc_in=None, unc_out=None, scales_device=None):
        B, J, W = self.B, self.J, self.W
        g = _ptrs([grads[b][j][w] for b in range(B) for j in range(J) for w in range(W)])
        e = _ptrs([errs[b][j][w] for b in range(B) for j in range(J) for w in range(W)])
        qq = _ptrs([q[b][j] for b in range(B) for j in range(J)])
        gh = _ptrs([ghat[b][j] for b in range(B) for j in range(J)])
        sc = (ctypes.c_float * B)(*[float(s) for s in scales]) if scales is not None else None
        ui = _ptrs([unc_in[b][w] for b in range(B) for w in range(W)]) if unc_in is not None else None
        uo = _ptrs([unc_out[b] for b in range(B)]) if unc_out is not None else None
        return psgd_step_args(g, e, qq, sc, gh, ui, uo, c_void_p(self.counts.data_ptr()),
                              c_void_p(self.skip.data_ptr()),
                              c_void_p(self.mask.data_ptr() if self.mask is not None else 0),
                              c_void_p(scales_device.data_ptr() if scales_device is not None else 0))

    def _stream(self):
        return self.torch.cuda.current_stream(self.device).cuda_stream

    def step(self, grads, errs, q, scales, ghat, unc_in=None, unc_out=None, scales_device=None):
        args = self._args(grads, errs, q, scales, ghat, unc_in, unc_out, scales_device)
        psgd_step(self.handle, args, self._stream())

    # Data-parallel exchange points (a handle made with PSGD_FLAG_EXCHANGE): step_p,
    # all-reduce (sum) of exchange_p() and exchange_counts(), step_q, all-reduce of
    # exchange_q(), step_e. The same arguments as step().
    def step_p(self, grads, errs, q, scales, ghat, scales_device=None):
        args = self._args(grads, errs, q, scales, ghat, scales_device=scales_device)
        psgd_step_p(self.handle, args, self._stream())

    def step_q(self, grads, errs, q, scales, ghat, block_counts, total_workers, scales_device=None):
        args = self._args(grads, errs, q, scales, ghat, scales_device=scales_device)
        psgd_step_q(self.handle, args, block_counts.data_ptr(), total_workers, self._stream())

    def step_e(self, grads, errs, q, scales, ghat, total_workers, scales_device=None):
        args = self._args(grads, errs, q, scales, ghat, scales_device=scales_device)
        psgd_step_e(self.handle, args, total_workers, self._stream())

    def _ws_view(self, ptr, count, dtype):
        es = self.torch.empty((), dtype=dtype).element_size()
        off = ptr - self.workspace.data_ptr()
        return self.workspace[off:off + count * es].view(dtype)

    def exchange_p(self):
        """The P exchange buffers of every matrix, one flat fp32 view in (b, j) order."""
        n = self.B * sum(m for m, _ in self.shapes) * self.r
        return self._ws_view(psgd_exchange_p(self.handle, 0, 0), n, self.torch.float32)

    def exchange_q(self):
        """The Q exchange buffers of every matrix, one flat fp32 view in (b, j) order."""
        n = self.B * sum(c for _, c in self.shapes) * self.r
        return self._ws_view(psgd_exchange_q(self.handle, 0, 0), n, self.torch.float32)

    def exchange_counts(self):
        """This rank's per-block nonfinite counts (int64 [B]), written by step_p."""
        return self._ws_view(psgd_exchange_counts(self.handle), self.B, self.torch.int64)

    def check(self):
        psgd_check(self.handle, self.torch.cuda.current_stream(self.device).cuda_stream)

    def debug_m(self, b, j, w, dtype):
        """A torch view of M_{b,j,w} in the workspace (valid until the next step)."""
        ptr = lib.psgd_debug_m(c_void_p(self.handle), b, j, w)
        m, n = self.shapes[j]
        es = self.torch.empty((), dtype=dtype).element_size()
        off = ptr - self.workspace.data_ptr()
        return self.workspace[off:off + m * n * es].view(dtype).view(m, n)

    def debug_phat(self, b, j):
        ptr = lib.psgd_debug_phat(c_void_p(self.handle), b, j)
        m, _ = self.shapes[j]
        rp = (self.r + 15) // 16 * 16
        off = ptr - self.workspace.data_ptr()
        return self.workspace[off:off + m * rp * 4].view(self.torch.float32).view(m, rp)[:, :self.r]

    def debug_orth(self, b, j):
        """(passes run in the last step, per-pass records [final, buffer, shifted, dead])."""
        out = (c_int32 * (4 * PSGD_MAX_ORTH_PASSES))()
        n = lib.psgd_debug_orth(c_void_p(self.handle), b, j, out,
                                c_void_p(self.torch.cuda.current_stream(self.device).cuda_stream))
        if n < 0:
            raise PSGDError(PSGD_EINVAL, "psgd_debug_orth failed")
        return n, [list(out[4 * k:4 * k + 4]) for k in range(PSGD_MAX_ORTH_PASSES)]

    def close(self):
        if getattr(self, "handle", None):
            psgd_finalize(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
