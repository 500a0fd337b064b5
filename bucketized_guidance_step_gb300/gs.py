"""Python binding of ``libgs.so`` (ctypes): argument marshalling only.

Every function here maps one-to-one onto an entry point of ``include/gs.h``;
all arithmetic of the step happens in the library (host C++ for the schedule
and the bucket plan, CUDA kernels for the mask and the step).  Torch is used
for device memory and streams: tensors are passed by data pointer and work is
enqueued on ``torch.cuda.current_stream()``.

The library is loaded on first use.  If it is missing or does not load, every
call raises ``GSLibraryError``; there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgs.so")
_lib = None
_lock = threading.Lock()

# ---- constants mirrored from include/gs.h ---------------------------------
GS_OK, GS_ERR_INVALID_ARG, GS_ERR_UNSUPPORTED, GS_ERR_CUDA = 0, 1, 2, 3
GS_ERR_STEP_RANGE, GS_ERR_NEED_UNCOND, GS_ERR_SIGMA, GS_ERR_CAPACITY = 4, 5, 6, 7
GS_ERR_TIMEOUT = 8
GS_DEV_STEP_RANGE, GS_DEV_NEED_UNCOND, GS_DEV_SIGMA, GS_DEV_TIMEOUT = 1, 2, 4, 8
GS_DTYPE_F32, GS_DTYPE_BF16, GS_DTYPE_F16 = 0, 1, 2
GS_SCHED_KARRAS, GS_SCHED_NORMAL = 0, 1
GS_CURVE_LINEAR, GS_CURVE_STEP, GS_CURVE_TABLE, GS_CURVE_PEAK = 0, 1, 2, 3
GS_MAX_REGIONS = 16
GS_LAUNCH_PDL = 1
GS_LAUNCH_NO_TMA = 2
GS_LAUNCH_TEST_WAIT_TIMEOUT = 4
GS_ABI_VERSION = 6
GS_STEP_PLAN_BYTES = 8192

EXPORTS = ("gs_sigmas", "gs_bucket_plan", "gs_mask_prepare", "gs_mask_rows", "gs_mask_spans",
           "gs_guided_step", "gs_step_prepare", "gs_step_launch",
           "gs_areas_to_latent", "gs_pack_conds",
           "gs_step_kernel_kind", "gs_status_from_word", "gs_status_string", "gs_abi_version")
GS_KERNEL_SCALAR, GS_KERNEL_VECTOR, GS_KERNEL_TMA = 0, 1, 2
KERNEL_NAMES = {0: "scalar", 1: "vector", 2: "tma"}
SAMPLERS = {"euler": 0, "euler_ancestral": 1}


class GSLibraryError(RuntimeError):
    """libgs.so is missing or could not be loaded."""


class GSError(RuntimeError):
    """An entry point returned a status other than GS_OK."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


# ---- struct mirrors ---------------------------------------------------------
class ScheduleDesc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("steps", ctypes.c_int32),
                ("sigma_min", ctypes.c_double), ("sigma_max", ctypes.c_double),
                ("rho", ctypes.c_double), ("denoise", ctypes.c_double),
                ("start_step", ctypes.c_int32), ("last_step", ctypes.c_int32),
                ("force_full_denoise", ctypes.c_int32), ("n_train", ctypes.c_int32),
                ("beta_start", ctypes.c_double), ("beta_end", ctypes.c_double)]


class CurveDesc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("v0", ctypes.c_double), ("v1", ctypes.c_double),
                ("edge", ctypes.c_double), ("interp", ctypes.c_int32)]


class RegionDesc(ctypes.Structure):
    _fields_ = [("y0", ctypes.c_int32), ("x0", ctypes.c_int32), ("h", ctypes.c_int32),
                ("w", ctypes.c_int32), ("strength", ctypes.c_float), ("feather", ctypes.c_int32),
                ("mask", ctypes.c_void_p), ("mask_bstride", ctypes.c_int64),
                ("out", ctypes.c_void_p), ("pitch", ctypes.c_int64),
                ("t_start", ctypes.c_double), ("t_end", ctypes.c_double),
                ("negative", ctypes.c_int32)]


class Area(ctypes.Structure):
    _fields_ = [("units", ctypes.c_int32), ("y0", ctypes.c_double), ("x0", ctypes.c_double),
                ("h", ctypes.c_double), ("w", ctypes.c_double)]


class Rect(ctypes.Structure):
    _fields_ = [("y0", ctypes.c_int32), ("x0", ctypes.c_int32), ("h", ctypes.c_int32),
                ("w", ctypes.c_int32)]


class CondEntry(ctypes.Structure):
    _fields_ = [("h", ctypes.c_int32), ("w", ctypes.c_int32), ("rows", ctypes.c_int32),
                ("options", ctypes.c_int64)]


class CondChunk(ctypes.Structure):
    _fields_ = [("call", ctypes.c_int32), ("entry", ctypes.c_int32), ("row0", ctypes.c_int32),
                ("rows", ctypes.c_int32)]


class StepArgs(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("C", ctypes.c_int32), ("H", ctypes.c_int32),
                ("W", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("x", ctypes.c_void_p), ("x_out", ctypes.c_void_p),
                ("denoised_out", ctypes.c_void_p),
                ("uncond", ctypes.c_void_p), ("cond", ctypes.c_void_p),
                ("n_regions", ctypes.c_int32), ("regions", ctypes.POINTER(RegionDesc)),
                ("sigmas", ctypes.c_void_p), ("n_sigmas", ctypes.c_int32),
                ("step_idx", ctypes.c_void_p), ("step", ctypes.c_int32),
                ("scale_lut", ctypes.c_void_p), ("n_lut", ctypes.c_int32),
                ("cfg", ctypes.c_float),
                ("inpaint_mask", ctypes.c_void_p), ("mask_bstride", ctypes.c_int64),
                ("mask_present", ctypes.c_void_p), ("original", ctypes.c_void_p),
                ("dev_status", ctypes.c_void_p), ("launch_flags", ctypes.c_uint32),
                ("mask_rows", ctypes.c_void_p),
                ("sampler", ctypes.c_int32), ("noise", ctypes.c_void_p),
                ("model_in_out", ctypes.c_void_p), ("orig_noise", ctypes.c_void_p),
                ("mask_spans", ctypes.c_void_p), ("unit_scale_skip", ctypes.c_int32)]


class StepPlan(ctypes.Structure):
    """gs_step_plan: a prepared launch (opaque, caller-owned host memory)."""
    _fields_ = [("opaque", ctypes.c_uint64 * (GS_STEP_PLAN_BYTES // 8))]


def library_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load libgs.so once; raise GSLibraryError if it is not there."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise GSLibraryError(f"{_LIB_PATH} is missing: build it with "
                                 "`python -m bucketized_guidance_step_gb300.build`")
        try:
            lib = ctypes.CDLL(_LIB_PATH)
        except OSError as e:  # pragma: no cover - depends on the host
            raise GSLibraryError(f"cannot load {_LIB_PATH}: {e}") from e
        i32, p = ctypes.c_int32, ctypes.c_void_p
        lib.gs_sigmas.argtypes = [ctypes.POINTER(ScheduleDesc), p, i32, p, p]
        lib.gs_bucket_plan.argtypes = [i32, i32, ctypes.POINTER(CurveDesc), p, p, p]
        lib.gs_mask_prepare.argtypes = [p, i32, i32, i32, p, i32, i32, p]
        lib.gs_mask_rows.argtypes = [p, i32, i32, i32, p, p]
        lib.gs_mask_spans.argtypes = [p, i32, i32, i32, p, p]
        lib.gs_guided_step.argtypes = [ctypes.POINTER(StepArgs), p]
        lib.gs_step_kernel_kind.argtypes = [ctypes.POINTER(StepArgs), p]
        lib.gs_step_prepare.argtypes = [ctypes.POINTER(StepArgs), ctypes.POINTER(StepPlan)]
        lib.gs_step_launch.argtypes = [ctypes.POINTER(StepPlan), i32, p]
        lib.gs_status_from_word.argtypes = [ctypes.c_uint32]
        lib.gs_status_string.argtypes = [i32]
        lib.gs_status_string.restype = ctypes.c_char_p
        lib.gs_abi_version.argtypes = []
        lib.gs_areas_to_latent.argtypes = [ctypes.POINTER(Area), i32, i32, i32, i32,
                                           ctypes.POINTER(Rect)]
        lib.gs_pack_conds.argtypes = [ctypes.POINTER(CondEntry), i32, ctypes.c_int64,
                                      ctypes.POINTER(CondChunk), i32, p, p]
        for f in ("gs_sigmas", "gs_bucket_plan", "gs_mask_prepare", "gs_mask_rows", "gs_mask_spans",
                  "gs_guided_step", "gs_step_prepare", "gs_step_launch",
                  "gs_step_kernel_kind", "gs_status_from_word", "gs_abi_version",
                  "gs_areas_to_latent", "gs_pack_conds"):
            getattr(lib, f).restype = i32
        if lib.gs_abi_version() != GS_ABI_VERSION:
            raise GSLibraryError("libgs.so ABI version does not match the binding")
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().gs_status_string(int(status)).decode()


def status_from_word(word: int) -> int:
    return int(load().gs_status_from_word(int(word) & 0xFFFFFFFF))


def _check(fn: str, status: int) -> None:
    if status != GS_OK:
        raise GSError(fn, status)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ---- host entry points --------------------------------------------------------
def sigmas(kind: str, steps: int, *, sigma_min: float = 0.0292, sigma_max: float = 14.6146,
           rho: float = 7.0, denoise: float = 1.0, start_step: int = -1, last_step: int = -1,
           force_full_denoise: bool = False, n_train: int = 1000, beta_start: float = 0.00085,
           beta_end: float = 0.012) -> Tuple[np.ndarray, int]:
    """gs_sigmas: the schedule as float32 and the offset of its first value in the base."""
    lib = load()
    d = ScheduleDesc(GS_SCHED_KARRAS if kind == "karras" else
                     GS_SCHED_NORMAL if kind == "normal" else -1,
                     int(steps), sigma_min, sigma_max, rho, denoise, int(start_step),
                     int(last_step), int(bool(force_full_denoise)), int(n_train),
                     beta_start, beta_end)
    n = ctypes.c_int32(0)
    off = ctypes.c_int32(0)
    st = lib.gs_sigmas(ctypes.byref(d), None, 0, ctypes.byref(n), ctypes.byref(off))
    if st not in (GS_OK, GS_ERR_CAPACITY):
        _check("gs_sigmas", st)
    out = np.zeros(max(n.value, 1), dtype=np.float32)
    _check("gs_sigmas", lib.gs_sigmas(ctypes.byref(d), _ptr(out), out.size, ctypes.byref(n),
                                      ctypes.byref(off)))
    return out[: n.value].copy(), off.value


AREA_UNITS = {"latent": 0, "pixels": 1, "fraction": 2}


def areas_to_latent(areas: Sequence[Tuple[str, float, float, float, float]], H: int, W: int,
                    scale: int = 8) -> List[Tuple[int, int, int, int]]:
    """gs_areas_to_latent: (units, y0, x0, h, w) areas -> (y0, x0, h, w) latent slices
    covering them, clipped to H x W ((0, 0, 0, 0) for an area that covers no pixel).
    units: "latent", "pixels" (divided by the VAE scale) or "fraction" (of H and W)."""
    n = len(areas)
    arr = (Area * max(n, 1))()
    for i, (u, y0, x0, h, w) in enumerate(areas):
        if u not in AREA_UNITS:
            raise ValueError(f"unknown area units {u!r}")
        arr[i] = Area(AREA_UNITS[u], float(y0), float(x0), float(h), float(w))
    out = (Rect * max(n, 1))()
    _check("gs_areas_to_latent", load().gs_areas_to_latent(arr, n, int(H), int(W), int(scale),
                                                           out))
    return [(r.y0, r.x0, r.h, r.w) for r in out[:n]]


def pack_conds(entries: Sequence[Tuple[int, int, int, int]], budget: int
               ) -> Tuple[int, List[Tuple[int, int, int, int]]]:
    """gs_pack_conds: cond entries (h, w, rows, options) -> (number of model calls,
    chunks (call, entry, row0, rows)); budget = latent pixels per call."""
    lib = load()
    n = len(entries)
    arr = (CondEntry * max(n, 1))()
    for i, (h, w, rows, opt) in enumerate(entries):
        arr[i] = CondEntry(int(h), int(w), int(rows), int(opt))
    nch, ncall = ctypes.c_int32(0), ctypes.c_int32(0)
    cap = max(n, 1)
    while True:
        chunks = (CondChunk * cap)()
        st = lib.gs_pack_conds(arr, n, int(budget), chunks, cap, ctypes.byref(nch),
                               ctypes.byref(ncall))
        if st == GS_ERR_CAPACITY:
            cap = nch.value
            continue
        _check("gs_pack_conds", st)
        return ncall.value, [(c.call, c.entry, c.row0, c.rows) for c in chunks[:nch.value]]


def bucket_plan(steps: int, num_buckets: int, *, curve: str = "linear", v0: float = 0.0,
                v1: float = 0.0, edge: float = 0.0, interp: bool = False,
                table: Optional[Sequence[float]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """gs_bucket_plan: per-step bucket ids (int32) and scales (float32).

    curve: "linear" (v0 -> v1), "step" (v0 before progress edge, v1 after), "peak"
    (v1 at both ends, v0 at progress edge) or "table"; interp: linear interpolation
    inside each bucket between the curve's values at its edges."""
    lib = load()
    kind = {"linear": GS_CURVE_LINEAR, "step": GS_CURVE_STEP, "table": GS_CURVE_TABLE,
            "peak": GS_CURVE_PEAK}.get(curve, -1)
    c = CurveDesc(kind, v0, v1, edge, 1 if interp else 0)
    tab = None if table is None else np.ascontiguousarray(table, dtype=np.float64)
    ids = np.zeros(max(int(steps), 1), dtype=np.int32)
    lut = np.zeros(max(int(steps), 1), dtype=np.float32)
    _check("gs_bucket_plan", lib.gs_bucket_plan(int(steps), int(num_buckets), ctypes.byref(c),
                                                None if tab is None else _ptr(tab),
                                                _ptr(ids), _ptr(lut)))
    return ids[:steps], lut[:steps]


# ---- device entry points ------------------------------------------------------
def _torch():
    import torch
    return torch


def _stream_ptr(stream=None) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _dptr(t, name: str, dtype=None) -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return int(t.data_ptr())


def mask_prepare(pix_mask, H: int, W: int, out=None, stream=None):
    """gs_mask_prepare: [B,1,Hp,Wp] fp32 pixel mask -> [B,1,H,W] fp32 latent mask."""
    torch = _torch()
    B, one, Hp, Wp = pix_mask.shape
    if one != 1:
        raise ValueError("pixel mask must have one channel")
    if out is None:
        out = torch.empty((B, 1, H, W), dtype=torch.float32, device=pix_mask.device)
    _check("gs_mask_prepare", load().gs_mask_prepare(
        _dptr(pix_mask, "pix_mask", torch.float32), B, Hp, Wp,
        _dptr(out, "out", torch.float32), int(H), int(W), _stream_ptr(stream)))
    return out


def mask_rows(lat_mask, out=None, stream=None):
    """gs_mask_rows: [Bm,1,H,W] fp32 latent mask -> [Bm, ceil(H/32)] int32 words whose
    bit (y mod 32) of word y // 32 says whether row y holds any nonzero value (the
    bits of a uint32, stored as int32)."""
    torch = _torch()
    Bm, one, H, W = lat_mask.shape
    if one != 1:
        raise ValueError("latent mask must have one channel")
    words = (H + 31) // 32
    if out is None:
        out = torch.empty((Bm, words), dtype=torch.int32, device=lat_mask.device)
    elif tuple(out.shape) != (Bm, words):
        raise ValueError(f"out must be [{Bm}, {words}]")
    _check("gs_mask_rows", load().gs_mask_rows(
        _dptr(lat_mask, "lat_mask", torch.float32), Bm, H, W, _dptr(out, "out", torch.int32),
        _stream_ptr(stream)))
    return out


def mask_spans(lat_mask, out=None, stream=None):
    """gs_mask_spans: [Bm,1,H,W] fp32 latent mask -> [Bm, H] int32 words, word y of mask
    b = lo | hi << 16 with [lo, hi) its row's nonzero column span (0: no nonzero value;
    the bits of a uint32, stored as int32)."""
    torch = _torch()
    Bm, one, H, W = lat_mask.shape
    if one != 1:
        raise ValueError("latent mask must have one channel")
    if out is None:
        out = torch.empty((Bm, H), dtype=torch.int32, device=lat_mask.device)
    elif tuple(out.shape) != (Bm, H):
        raise ValueError(f"out must be [{Bm}, {H}]")
    _check("gs_mask_spans", load().gs_mask_spans(
        _dptr(lat_mask, "lat_mask", torch.float32), Bm, H, W, _dptr(out, "out", torch.int32),
        _stream_ptr(stream)))
    return out


@dataclass
class Region:
    """One regional conditioning output for ``guided_step`` (see gs_region)."""
    y0: int
    x0: int
    h: int
    w: int
    strength: float
    feather: int
    out: object                       # CUDA tensor [B, C, h, pitch], the latent dtype
    mask: object = None               # CUDA fp32 [h, w] or [B, h, w], or None
    pitch: Optional[int] = None       # defaults to out.shape[-1]
    t_start: float = 0.0              # timestep range [t_start, t_end) in progress i/S;
    t_end: float = 0.0                # t_end <= t_start: every step
    negative: bool = False            # part of the uncond branch (regional uncond)


_DT = {}


def _dtype_code(t) -> int:
    torch = _torch()
    if not _DT:
        _DT.update({torch.float32: GS_DTYPE_F32, torch.bfloat16: GS_DTYPE_BF16,
                    torch.float16: GS_DTYPE_F16})
    if t.dtype not in _DT:
        raise ValueError(f"unsupported latent dtype {t.dtype}")
    return _DT[t.dtype]


def make_step_args(x, *, sigmas, uncond=None, cond=None, stacked=None, step_idx=None,
                   step: int = 0, scale_lut=None, cfg: float = 1.0,
                   regions: Sequence[Region] = (), inpaint_mask=None, mask_present=None,
                   original=None, mask_rows=None, mask_spans=None, unit_scale_skip=False,
                   x_out=None, denoised_out=None, status=None,
                   sampler: str = "euler", noise=None, model_in_out=None, orig_noise=None,
                   pdl: bool = False, tma: bool = True, test_wait_timeout: bool = False):
    """Build a gs_step_args (and the region array it points to) from tensors."""
    torch = _torch()
    B, C, H, W = x.shape
    if stacked is not None:
        if uncond is not None or cond is not None:
            raise ValueError("pass either stacked or uncond/cond")
        if stacked.shape[0] != 2 * B:
            raise ValueError("stacked must be [2B, C, H, W]")
        uncond, cond = stacked[:B], stacked[B:]
    dt = x.dtype
    shape = tuple(x.shape)
    for name, t in (("x_out", x_out), ("denoised_out", denoised_out), ("uncond", uncond),
                    ("cond", cond), ("original", original), ("noise", noise),
                    ("model_in_out", model_in_out), ("orig_noise", orig_noise)):
        if t is not None and tuple(t.shape) != shape:
            raise ValueError(f"{name} must have the shape of x {shape}, got {tuple(t.shape)}")
    if inpaint_mask is not None and (inpaint_mask.dim() != 4 or inpaint_mask.shape[0] not in (1, B)
                                     or tuple(inpaint_mask.shape[1:]) != (1, H, W)):
        raise ValueError("inpaint_mask must be [1 or B, 1, H, W]")
    if mask_present is not None and tuple(mask_present.shape) != (B,):
        raise ValueError("mask_present must be [B]")
    if step_idx is not None and tuple(step_idx.shape) != (B,):
        raise ValueError("step_idx must be [B]")
    if status is not None and status.numel() < 1:
        raise ValueError("status needs one element")
    reg_arr = (RegionDesc * max(len(regions), 1))()
    for i, r in enumerate(regions):
        pitch = int(r.pitch if r.pitch is not None else r.out.shape[-1])
        if r.out.dim() != 4 or tuple(r.out.shape[:3]) != (B, C, r.h) or r.out.shape[3] < r.w \
                or r.out.shape[3] != pitch:
            raise ValueError(f"region {i}: out must be [B, C, h, pitch >= w]")
        mstride = 0
        if r.mask is not None:
            if tuple(r.mask.shape[-2:]) != (r.h, r.w) or r.mask.dim() not in (2, 3) or \
                    (r.mask.dim() == 3 and r.mask.shape[0] not in (1, B)):
                raise ValueError(f"region {i}: mask must be [h, w] or [B, h, w]")
            if r.mask.dim() == 3 and r.mask.shape[0] == B:
                mstride = r.h * r.w
        reg_arr[i] = RegionDesc(int(r.y0), int(r.x0), int(r.h), int(r.w), float(r.strength),
                                int(r.feather), _dptr(r.mask, "region mask", torch.float32),
                                mstride, _dptr(r.out, "region out", dt), pitch,
                                float(r.t_start), float(r.t_end), int(bool(r.negative)))
    mstride = 0
    if inpaint_mask is not None:
        mstride = 0 if inpaint_mask.shape[0] == 1 else H * W
    a = StepArgs()
    a.B, a.C, a.H, a.W = int(B), int(C), int(H), int(W)
    a.dtype = _dtype_code(x)
    a.x = _dptr(x, "x", dt)
    a.x_out = _dptr(x if x_out is None else x_out, "x_out", dt)
    a.denoised_out = _dptr(denoised_out, "denoised_out", dt)
    a.uncond = _dptr(uncond, "uncond", dt)
    a.cond = _dptr(cond, "cond", dt)
    a.n_regions = len(regions)
    a.regions = ctypes.cast(reg_arr, ctypes.POINTER(RegionDesc))
    a.sigmas = _dptr(sigmas, "sigmas", torch.float32)
    a.n_sigmas = int(sigmas.numel())
    a.step_idx = _dptr(step_idx, "step_idx", torch.int32)
    a.step = int(step)
    a.scale_lut = _dptr(scale_lut, "scale_lut", torch.float32)
    a.n_lut = 0 if scale_lut is None else int(scale_lut.numel())
    a.cfg = float(cfg)
    a.inpaint_mask = _dptr(inpaint_mask, "inpaint_mask", torch.float32)
    a.mask_bstride = mstride
    a.mask_present = _dptr(mask_present, "mask_present", torch.uint8)
    a.original = _dptr(original, "original", dt)
    a.dev_status = _dptr(status, "status", torch.int32)
    if mask_rows is not None:
        if inpaint_mask is None:
            raise ValueError("mask_rows needs inpaint_mask")
        if tuple(mask_rows.shape) != (inpaint_mask.shape[0], (H + 31) // 32):
            raise ValueError("mask_rows must be [masks, ceil(H/32)] (from mask_rows())")
    a.mask_rows = _dptr(mask_rows, "mask_rows", torch.int32)
    if mask_spans is not None:
        if inpaint_mask is None:
            raise ValueError("mask_spans needs inpaint_mask")
        if tuple(mask_spans.shape) != (inpaint_mask.shape[0], H):
            raise ValueError("mask_spans must be [masks, H] (from mask_spans())")
    a.mask_spans = _dptr(mask_spans, "mask_spans", torch.int32)
    a.unit_scale_skip = 1 if unit_scale_skip else 0
    if sampler not in SAMPLERS:
        raise ValueError(f"sampler must be one of {tuple(SAMPLERS)}")
    if sampler == "euler_ancestral" and noise is None:
        raise ValueError("the ancestral sampler needs noise")
    if model_in_out is not None and (inpaint_mask is None or orig_noise is None):
        raise ValueError("model_in_out needs inpaint_mask, original and orig_noise")
    a.sampler = SAMPLERS[sampler]
    a.noise = _dptr(noise, "noise", dt)
    a.model_in_out = _dptr(model_in_out, "model_in_out", dt)
    a.orig_noise = _dptr(orig_noise, "orig_noise", dt)
    a.launch_flags = ((GS_LAUNCH_PDL if pdl else 0) | (0 if tma else GS_LAUNCH_NO_TMA) |
                      (GS_LAUNCH_TEST_WAIT_TIMEOUT if test_wait_timeout else 0))
    return a, reg_arr


def launch_step(args: StepArgs, stream=None) -> None:
    """gs_guided_step on prepared arguments (the lowest-overhead call)."""
    _check("gs_guided_step", load().gs_guided_step(ctypes.byref(args), _stream_ptr(stream)))


def prepare_step(args: StepArgs) -> StepPlan:
    """gs_step_prepare: check prepared arguments once and build the launch (the
    tensors behind the arguments must stay alive while the plan is used)."""
    plan = StepPlan()
    _check("gs_step_prepare", load().gs_step_prepare(ctypes.byref(args), ctypes.byref(plan)))
    return plan


def launch_prepared(plan: StepPlan, step: int = 0, stream=None) -> None:
    """gs_step_launch: one step from a plan (step: the shared step index when the plan
    was prepared without step_idx)."""
    _check("gs_step_launch", load().gs_step_launch(ctypes.byref(plan), int(step),
                                                   _stream_ptr(stream)))


class StepLauncher:
    """A prepared step bound to one stream: ``launcher(step)`` launches one step
    (gs_step_launch) with the least Python work per call -- the plan, the stream handle
    and the library function are looked up once, here."""

    def __init__(self, plan: StepPlan, stream=None):
        self._fn = load().gs_step_launch
        self._plan = plan                       # keeps the plan alive
        self._ref = ctypes.byref(plan)
        self._stream = ctypes.c_void_p(_stream_ptr(stream))

    def __call__(self, step: int = 0) -> None:
        status = self._fn(self._ref, step, self._stream)
        if status != GS_OK:
            raise GSError("gs_step_launch", status)


def kernel_kind(args: StepArgs) -> str:
    """gs_step_kernel_kind: "tma", "vector" or "scalar" for prepared arguments."""
    k = ctypes.c_int32(-1)
    _check("gs_step_kernel_kind", load().gs_step_kernel_kind(ctypes.byref(args), ctypes.byref(k)))
    return KERNEL_NAMES[k.value]


def guided_step(x, *, sigmas, stream=None, **kw):
    """gs_guided_step: one fused guided denoise step; returns x_out (x itself by default).

    Keyword arguments follow gs_step_args: uncond / cond or stacked, regions,
    step_idx (int32 [B]) or step, scale_lut (fp32) or cfg, inpaint_mask
    ([B or 1, 1, H, W] fp32), mask_present (uint8 [B]), original, x_out,
    denoised_out, status (int32 [1], device flags OR-ed in), mask_rows (the row
    summary of inpaint_mask from ``mask_rows()``: bands whose mask is 0 on every row
    then skip reading the prediction), mask_spans (the span summary from
    ``mask_spans()``: also narrows the prediction reads to the nonzero columns),
    unit_scale_skip (samples of scale exactly 1 read no uncond), sampler ("euler" or "euler_ancestral"), noise
    (the ancestral step's fresh noise), model_in_out and orig_noise (the next model
    input under the inpaint wrapper), pdl, tma (False forces the register-streaming
    kernel).
    """
    args, _keep = make_step_args(x, sigmas=sigmas, **kw)
    launch_step(args, stream)
    return x if kw.get("x_out") is None else kw["x_out"]
