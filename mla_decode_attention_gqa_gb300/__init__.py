"""Python binding of libsplitkv_attn.so: exact split-KV attention with an LSE merge on GB300.

Thin ctypes marshalling over the C ABI declared in ``include/splitkv_attn.h``:
every step of the computation runs in the library's CUDA kernels; PyTorch only
provides device memory (outputs, workspace) and the current CUDA stream.  There is
no CPU fallback: the first call loads the library and raises if it is missing, and
every call fails if its tensors are not on a CUDA device.

split_bounds is an int32 tensor [B, n_split + 1] on the call's device (the C ABI reads
it in device memory); a nested list is accepted and copied to the device at each call.

Entry points (same names as the C ABI):
  attn_partial(q, k_cache, v_cache, seq_lens, split_bounds, ...) -> (out_partial, lse_partial)
  attn_merge_lse(out_partials, lse_partials) -> (out, lse)
  gqa_decode_attn(q, k_cache, v_cache, seq_lens, split_bounds, ...) -> (out, lse)
  gqa_decode_attn_noalloc(...) -> (out, lse)   (no workspace: the library's own scratch)
  gqa_decode_attn_passq(q, k_shards, v_shards, shard_lens, ...) -> (out, lse)
plus the position-masked (_pos), paged (_paged) and pass-KV ring-step variants.
"""

import ctypes
import functools
import inspect
import math
import os

import torch

from .workloads import NO_CAUSAL

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsplitkv_attn.so")

SKV_OK, SKV_EINVAL, SKV_EUNSUPPORTED, SKV_ECUDA, SKV_EWORKSPACE = 0, -1, -2, -3, -4
SKV_KV_BF16, SKV_KV_FP8_E4M3 = 0, 1
_STATUS = {0: "SKV_OK", -1: "SKV_EINVAL", -2: "SKV_EUNSUPPORTED", -3: "SKV_ECUDA", -4: "SKV_EWORKSPACE"}

# Every symbol declared in include/splitkv_attn.h.
EXPORTED_SYMBOLS = (
    "splitkv_version",
    "splitkv_last_error",
    "splitkv_device_error",
    "splitkv_device_error_detail",
    "splitkv_kernel_timing",
    "splitkv_kernel_timing_read",
    "attn_partial_workspace_size",
    "attn_partial",
    "attn_merge_lse",
    "gqa_decode_attn_workspace_size",
    "gqa_decode_attn",
    "gqa_decode_attn_noalloc",
    "attn_partial_pos",
    "gqa_decode_attn_pos",
    "attn_partial_paged",
    "gqa_decode_attn_paged",
    "attn_ring_step_workspace_size",
    "attn_ring_step",
    "gqa_decode_attn_passq_workspace_size",
    "gqa_decode_attn_passq",
)

# Every symbol declared in include/splitkv_attn_selftest.h (hardware self-tests).
SELFTEST_SYMBOLS = ("splitkv_selftest_umma_gemm",)


class SkvDesc(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32),
        ("Tq", ctypes.c_int32),
        ("Hq", ctypes.c_int32),
        ("Hkv", ctypes.c_int32),
        ("dk", ctypes.c_int32),
        ("dv", ctypes.c_int32),
        ("S_max", ctypes.c_int64),
        ("softmax_scale", ctypes.c_float),
        ("kv_dtype", ctypes.c_int32),
        ("scale_block", ctypes.c_int32),
        ("q_strides", ctypes.c_int64 * 3),
        ("k_strides", ctypes.c_int64 * 3),
        ("v_strides", ctypes.c_int64 * 3),
    ]


class SplitKVError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m mla_decode_attention_gqa_gb300.build` "
            "(or __graft_entry__.build())")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    D = ctypes.POINTER(SkvDesc)
    I32P = ctypes.POINTER(ctypes.c_int32)
    lib.splitkv_version.restype = I32
    lib.splitkv_last_error.restype = ctypes.c_char_p
    lib.splitkv_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.splitkv_device_error.restype = I32
    lib.splitkv_device_error_detail.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.splitkv_device_error_detail.restype = I32
    lib.splitkv_kernel_timing.argtypes = [I32]
    lib.splitkv_kernel_timing.restype = I32
    lib.splitkv_kernel_timing_read.argtypes = [ctypes.POINTER(ctypes.c_float), I32P]
    lib.splitkv_kernel_timing_read.restype = I32
    for name in ("attn_partial_workspace_size", "gqa_decode_attn_workspace_size"):
        f = getattr(lib, name)
        f.argtypes = [D, I32, ctypes.POINTER(SZ)]
        f.restype = I32
    # split_bounds is a device pointer, like seq_lens
    common = [D, P, P, P, P, P, P, P, I32, I64]
    lib.attn_partial.argtypes = common + [P, P, P, SZ, P]
    lib.attn_partial.restype = I32
    lib.gqa_decode_attn.argtypes = common + [P, P, P, SZ, P]
    lib.gqa_decode_attn.restype = I32
    lib.gqa_decode_attn_noalloc.argtypes = common + [P, P, P]
    lib.gqa_decode_attn_noalloc.restype = I32
    lib.attn_merge_lse.argtypes = [I32, I32, I32, I32, I32, P, P, P, P, P]
    lib.attn_merge_lse.restype = I32
    common_pos = [D, P, P, P, P, P, P, P, I32, P, P]  # q_pos, k_pos replace causal_offset
    lib.attn_partial_pos.argtypes = common_pos + [P, P, P, SZ, P]
    lib.attn_partial_pos.restype = I32
    lib.gqa_decode_attn_pos.argtypes = common_pos + [P, P, P, SZ, P]
    lib.gqa_decode_attn_pos.restype = I32
    common_paged = [D, ctypes.POINTER(SkvPaged), P, P, P, P, P, P, P, I32, I64]
    lib.attn_partial_paged.argtypes = common_paged + [P, P, P, SZ, P]
    lib.attn_partial_paged.restype = I32
    lib.gqa_decode_attn_paged.argtypes = common_paged + [P, P, P, SZ, P]
    lib.gqa_decode_attn_paged.restype = I32
    lib.attn_ring_step_workspace_size.argtypes = [D, ctypes.POINTER(SZ)]
    lib.attn_ring_step_workspace_size.restype = I32
    lib.attn_ring_step.argtypes = [D, P, P, P, P, P, P, I64, I32, P, P, P, SZ, P]
    lib.attn_ring_step.restype = I32
    lib.gqa_decode_attn_passq_workspace_size.argtypes = [D, I32, ctypes.POINTER(SZ)]
    lib.gqa_decode_attn_passq_workspace_size.restype = I32
    lib.gqa_decode_attn_passq.argtypes = [D, I32, P, P, P, P, P, P, P, P, P, SZ, P]
    lib.gqa_decode_attn_passq.restype = I32
    return lib


class _LazyLib:
    """Loads the shared library at first use (so that the pure-host modules of this
    package - workloads, roofline - import without it); a missing library raises."""

    _handle = None

    def __getattr__(self, name):
        if _LazyLib._handle is None:
            _LazyLib._handle = _load()
        return getattr(_LazyLib._handle, name)


_lib = _LazyLib()


def load_library():
    """Load (once) and return the ctypes handle of libsplitkv_attn.so."""
    _lib.splitkv_version  # noqa: B018 - forces the load
    return _LazyLib._handle


def version():
    v = _lib.splitkv_version()
    return (v >> 16, v & 0xFFFF)


def last_error():
    return _lib.splitkv_last_error().decode()


last_device_error_detail = None


def device_error():
    """Read and clear the device error record (blocking); 0 means no kernel gave up a wait.
    A nonzero code also leaves the record (block, thread, barrier, parity) in
    ``last_device_error_detail`` and prints it to stderr."""
    global last_device_error_detail
    rec = (ctypes.c_uint32 * 8)()
    _check(_lib.splitkv_device_error_detail(rec))
    code = int(rec[0])
    if code:
        last_device_error_detail = {"code": code, "block": int(rec[2]), "thread": int(rec[3]),
                                    "barrier_smem_addr": int(rec[4]), "parity": int(rec[5]) & 0xFF,
                                    "first_code": (int(rec[5]) >> 8) & 0xFF}
        import sys as _sys

        print(f"device error record: {last_device_error_detail}", file=_sys.stderr)
    return code


def _check(status):
    if status != SKV_OK:
        raise SplitKVError(status, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class SkvPaged(ctypes.Structure):
    _fields_ = [
        ("block_len", ctypes.c_int32),
        ("max_blocks", ctypes.c_int32),
        ("num_blocks", ctypes.c_int64),
        ("block_table", ctypes.c_void_p),
    ]


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("split-KV attention runs on CUDA tensors only (no CPU path)")


def _on_tensor_device(fn):
    """Run a call with its first tensor's device current: the library launches on the
    current device and stream, so every tensor of the call must live on that device."""

    first = next(iter(inspect.signature(fn).parameters))

    @functools.wraps(fn)
    def wrapped(*args, **kw):
        t = args[0] if args else kw.get(first)
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError("split-KV attention runs on CUDA tensors only (no CPU path)")
        with torch.cuda.device(t.device):
            return fn(*args, **kw)

    return wrapped


def _same_device(dev, **tensors):
    for name, t in tensors.items():
        if t is not None and t.device != dev:
            raise ValueError(f"{name} is on {t.device} but q on {dev}: every tensor of a call must be on one device")


def _out(t, shape, dtype, dev, name):
    """The caller's output buffer, checked (exact shape and dtype, contiguous, on dev), or a new one."""
    shape = tuple(int(x) for x in shape)
    if t is None:
        return torch.empty(shape, dtype=dtype, device=dev)
    if t.device != dev or t.dtype != dtype or tuple(t.shape) != shape or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {shape} on {dev}")
    return t


def _ws_arg(workspace, nbytes, dev):
    """(buffer, bytes) of the caller's workspace, or of the library's cached scratch."""
    if workspace is None:
        return _workspace(nbytes, dev), nbytes
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError(f"workspace must be a contiguous tensor on {dev}")
    return workspace, workspace.numel() * workspace.element_size()


def _check_lens(t, n, name):
    if t.dtype != torch.int32 or not t.is_contiguous() or tuple(t.shape) != (n,):
        raise ValueError(f"{name} must be contiguous int32 of shape ({n},)")


def _check_scales(scales, shape, layout):
    shape = tuple(int(x) for x in shape)
    for s in scales:
        if s is not None and (s.dtype != torch.float32 or not s.is_contiguous() or tuple(s.shape) != shape):
            raise ValueError(f"scales must be contiguous float32 {layout} = {shape}")


def _kv_dtype(k):
    if k.dtype == torch.bfloat16:
        return SKV_KV_BF16
    if k.dtype in (torch.uint8, torch.float8_e4m3fn):
        return SKV_KV_FP8_E4M3
    raise ValueError(f"unsupported KV dtype {k.dtype}: bf16 or e4m3 codes (uint8 / float8_e4m3fn)")


def make_desc(q, k_cache, v_cache, softmax_scale=None, scale_block=64):
    """Describe q [B,Tq,Hq,dk] and k/v caches [B,Hkv,S,d] (any strides, unit last dim)."""
    if q.dim() != 4 or k_cache.dim() != 4 or v_cache.dim() != 4:
        raise ValueError("q must be [B,Tq,Hq,dk] and caches [B,Hkv,S,d]")
    if q.dtype != torch.bfloat16:
        raise ValueError("q must be bf16")
    for t in (q, k_cache, v_cache):
        if t.stride(-1) != 1:
            raise ValueError("the head dim must be unit-stride")
    B, Tq, Hq, dk = q.shape
    Bk, Hkv, S, dk2 = k_cache.shape
    if Bk != B or dk2 != dk or v_cache.shape[:3] != k_cache.shape[:3]:
        raise ValueError("q / k_cache / v_cache shapes disagree")
    d = SkvDesc()
    d.B, d.Tq, d.Hq, d.Hkv, d.dk, d.dv = B, Tq, Hq, Hkv, dk, v_cache.shape[3]
    d.S_max = S
    d.softmax_scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(dk)
    d.kv_dtype = _kv_dtype(k_cache)
    d.scale_block = scale_block
    for i in range(3):
        d.q_strides[i] = q.stride(i)
        d.k_strides[i] = k_cache.stride(i)
        d.v_strides[i] = v_cache.stride(i)
    return d


def _bounds_tensor(split_bounds, B, dev):
    """The split bounds as the device int32 tensor [B, n_split + 1] the library reads.  A
    tensor is checked and passed as it is; a nested list ([B][n_split + 1], or one row
    shared by every sequence) is copied to the device here, once per call (pass a device
    tensor to keep host-to-device copies out of a hot loop)."""
    if isinstance(split_bounds, torch.Tensor):
        t = split_bounds
        if t.device != dev or t.dtype != torch.int32 or t.dim() != 2 or t.shape[0] != B or t.shape[1] < 2 \
                or not t.is_contiguous():
            raise ValueError(f"split_bounds must be a contiguous int32 tensor [B, n_split + 1] on {dev}")
        return t, int(t.shape[1]) - 1
    rows = [list(map(int, r)) for r in split_bounds]
    if len(rows) == 1 and B > 1:
        rows = rows * B
    if len(rows) != B or len({len(r) for r in rows}) != 1 or len(rows[0]) < 2:
        raise ValueError("split_bounds must be [B][n_split+1] (or one row shared by every sequence)")
    return torch.tensor(rows, dtype=torch.int32, device=dev), len(rows[0]) - 1


_ws_cache = {}


def _workspace(nbytes, device):
    """A reusable device scratch buffer of at least nbytes (torch allocation), one per
    (device, current stream): calls on different streams never share one."""
    if nbytes == 0:
        return None
    key = (device.index if device.index is not None else torch.cuda.current_device(),
           torch.cuda.current_stream(device).cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _prep(q, k_cache, v_cache, seq_lens, split_bounds, k_scale, v_scale, softmax_scale, scale_block):
    _require_cuda(q, k_cache, v_cache, seq_lens, k_scale, v_scale)
    _same_device(q.device, k_cache=k_cache, v_cache=v_cache, seq_lens=seq_lens, k_scale=k_scale, v_scale=v_scale)
    d = make_desc(q, k_cache, v_cache, softmax_scale, scale_block)
    _check_lens(seq_lens, d.B, "seq_lens")
    bounds, n_split = (None, 1) if split_bounds is None else _bounds_tensor(split_bounds, d.B, q.device)
    if d.kv_dtype == SKV_KV_FP8_E4M3 and scale_block > 0:
        _check_scales((k_scale, v_scale), (d.B, d.Hkv, -(-d.S_max // scale_block)), "[B, Hkv, ceil(S / scale_block)]")
    return d, bounds, n_split


def _prep_paged(q, k_pages, v_pages, seq_lens, split_bounds, block_table, k_scale, v_scale, softmax_scale,
                scale_block):
    """Descriptor of a paged cache: pages [num_blocks, Hkv, block_len, d], block table
    int32 [B, max_blocks]; S_max = max_blocks * block_len logical tokens per sequence."""
    _require_cuda(q, k_pages, v_pages, seq_lens, k_scale, v_scale, block_table)
    _same_device(q.device, k_pages=k_pages, v_pages=v_pages, seq_lens=seq_lens, k_scale=k_scale, v_scale=v_scale,
                 block_table=block_table)
    if block_table.dtype != torch.int32 or not block_table.is_contiguous() or block_table.dim() != 2:
        raise ValueError("block_table must be contiguous int32 [B, max_blocks]")
    if q.dim() != 4 or k_pages.dim() != 4 or v_pages.dim() != 4:
        raise ValueError("q must be [B,Tq,Hq,dk] and pages [num_blocks,Hkv,block_len,d]")
    for t in (q, k_pages, v_pages):
        if t.stride(-1) != 1:
            raise ValueError("the head dim must be unit-stride")
    B, Tq, Hq, dk = q.shape
    nb, Hkv, L, dk2 = k_pages.shape
    if dk2 != dk or v_pages.shape[:3] != k_pages.shape[:3] or block_table.shape[0] != B:
        raise ValueError("q / pages / block_table shapes disagree")
    _check_lens(seq_lens, B, "seq_lens")
    d = SkvDesc()
    d.B, d.Tq, d.Hq, d.Hkv, d.dk, d.dv = B, Tq, Hq, Hkv, dk, v_pages.shape[3]
    d.S_max = block_table.shape[1] * L
    d.softmax_scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(dk)
    d.kv_dtype = _kv_dtype(k_pages)
    d.scale_block = scale_block
    for i in range(3):
        d.q_strides[i] = q.stride(i)
        d.k_strides[i] = k_pages.stride(i)
        d.v_strides[i] = v_pages.stride(i)
    pg = SkvPaged()
    pg.block_len, pg.max_blocks, pg.num_blocks = L, block_table.shape[1], nb
    pg.block_table = block_table.data_ptr()
    bounds, n_split = _bounds_tensor(split_bounds, B, q.device)
    if d.kv_dtype == SKV_KV_FP8_E4M3 and scale_block > 0:
        _check_scales((k_scale, v_scale), (nb, Hkv, L // scale_block), "[num_blocks, Hkv, block_len / scale_block]")
    return d, pg, bounds, n_split


def attn_partial_workspace_size(desc, n_split):
    n = ctypes.c_size_t(0)
    _check(_lib.attn_partial_workspace_size(ctypes.byref(desc), n_split, ctypes.byref(n)))
    return int(n.value)


def gqa_decode_attn_workspace_size(desc, n_split):
    n = ctypes.c_size_t(0)
    _check(_lib.gqa_decode_attn_workspace_size(ctypes.byref(desc), n_split, ctypes.byref(n)))
    return int(n.value)


@_on_tensor_device
def attn_partial(q, k_cache, v_cache, seq_lens, split_bounds, causal_offset=NO_CAUSAL, k_scale=None,
                 v_scale=None, softmax_scale=None, scale_block=64, out_partial=None, lse_partial=None):
    """Per-split partial attention: returns (out_partial fp32 [n_split,B,Tq,Hq,dv], lse fp32 [n_split,B,Tq,Hq])."""
    d, bounds, n_split = _prep(q, k_cache, v_cache, seq_lens, split_bounds, k_scale, v_scale, softmax_scale,
                               scale_block)
    dev = q.device
    out_partial = _out(out_partial, (n_split, d.B, d.Tq, d.Hq, d.dv), torch.float32, dev, "out_partial")
    lse_partial = _out(lse_partial, (n_split, d.B, d.Tq, d.Hq), torch.float32, dev, "lse_partial")
    nbytes = attn_partial_workspace_size(d, n_split)
    ws = _workspace(nbytes, dev)
    _check(_lib.attn_partial(ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                             _ptr(seq_lens), _ptr(bounds), n_split, int(causal_offset), _ptr(out_partial),
                             _ptr(lse_partial), _ptr(ws), nbytes, _stream()))
    return out_partial, lse_partial


@_on_tensor_device
def attn_merge_lse(out_partials, lse_partials, out=None, lse=None):
    """Exact LSE merge over the first axis: returns (out bf16 [B,Tq,Hq,dv], lse fp32 [B,Tq,Hq])."""
    _require_cuda(out_partials, lse_partials)
    if out_partials.dtype != torch.float32 or lse_partials.dtype != torch.float32:
        raise ValueError("partials must be float32")
    if not (out_partials.is_contiguous() and lse_partials.is_contiguous()):
        raise ValueError("partials must be contiguous")
    if out_partials.dim() != 5 or tuple(lse_partials.shape) != tuple(out_partials.shape[:4]):
        raise ValueError("partials must be out [n_split,B,Tq,Hq,dv] and lse [n_split,B,Tq,Hq]")
    dev = out_partials.device
    _same_device(dev, lse_partials=lse_partials)
    n_split, B, Tq, Hq, dv = out_partials.shape
    out = _out(out, (B, Tq, Hq, dv), torch.bfloat16, dev, "out")
    lse = _out(lse, (B, Tq, Hq), torch.float32, dev, "lse")
    _check(_lib.attn_merge_lse(n_split, B, Tq, Hq, dv, _ptr(out_partials), _ptr(lse_partials), _ptr(out), _ptr(lse),
                               _stream()))
    return out, lse


@_on_tensor_device
def gqa_decode_attn(q, k_cache, v_cache, seq_lens, split_bounds, causal_offset=NO_CAUSAL, k_scale=None,
                    v_scale=None, softmax_scale=None, scale_block=64, out=None, lse=None, workspace=None):
    """Split-KV attention plus merge in one call: returns (out bf16 [B,Tq,Hq,dv], lse fp32 [B,Tq,Hq])."""
    d, bounds, n_split = _prep(q, k_cache, v_cache, seq_lens, split_bounds, k_scale, v_scale, softmax_scale,
                               scale_block)
    dev = q.device
    out = _out(out, (d.B, d.Tq, d.Hq, d.dv), torch.bfloat16, dev, "out")
    lse = _out(lse, (d.B, d.Tq, d.Hq), torch.float32, dev, "lse")
    ws, ws_bytes = _ws_arg(workspace, gqa_decode_attn_workspace_size(d, n_split), dev)
    _check(_lib.gqa_decode_attn(ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                _ptr(seq_lens), _ptr(bounds), n_split, int(causal_offset), _ptr(out), _ptr(lse), _ptr(ws),
                                ws_bytes, _stream()))
    return out, lse


@_on_tensor_device
def gqa_decode_attn_noalloc(q, k_cache, v_cache, seq_lens, split_bounds, causal_offset=NO_CAUSAL, k_scale=None,
                            v_scale=None, softmax_scale=None, scale_block=64, out=None, lse=None):
    """gqa_decode_attn without a workspace: the library keeps the partials in a fixed scratch
    array of its own (32 MiB per device; calls that overlap on the GPU race for it)."""
    d, bounds, n_split = _prep(q, k_cache, v_cache, seq_lens, split_bounds, k_scale, v_scale, softmax_scale,
                               scale_block)
    dev = q.device
    out = _out(out, (d.B, d.Tq, d.Hq, d.dv), torch.bfloat16, dev, "out")
    lse = _out(lse, (d.B, d.Tq, d.Hq), torch.float32, dev, "lse")
    _check(_lib.gqa_decode_attn_noalloc(ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                        _ptr(v_scale), _ptr(seq_lens), _ptr(bounds), n_split, int(causal_offset),
                                        _ptr(out), _ptr(lse), _stream()))
    return out, lse


def _positions(q_pos, k_pos, d, dev):
    _require_cuda(q_pos, k_pos)
    _same_device(dev, q_pos=q_pos, k_pos=k_pos)
    for t, shape, name in ((q_pos, (d.B, d.Tq), "q_pos"), (k_pos, (d.B, d.S_max), "k_pos")):
        if t.dtype != torch.int32 or not t.is_contiguous() or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be contiguous int32 of shape {shape}")


@_on_tensor_device
def attn_partial_pos(q, k_cache, v_cache, seq_lens, split_bounds, q_pos, k_pos, k_scale=None, v_scale=None,
                     softmax_scale=None, scale_block=64, out_partial=None, lse_partial=None):
    """attn_partial with the causal rule taken from original positions: token t is visible to
    row i iff k_pos[b, t] <= q_pos[b, i] (q_pos int32 [B,Tq], k_pos int32 [B,S], on the GPU)."""
    d, bounds, n_split = _prep(q, k_cache, v_cache, seq_lens, split_bounds, k_scale, v_scale, softmax_scale,
                               scale_block)
    _positions(q_pos, k_pos, d, q.device)
    dev = q.device
    out_partial = _out(out_partial, (n_split, d.B, d.Tq, d.Hq, d.dv), torch.float32, dev, "out_partial")
    lse_partial = _out(lse_partial, (n_split, d.B, d.Tq, d.Hq), torch.float32, dev, "lse_partial")
    nbytes = attn_partial_workspace_size(d, n_split)
    ws = _workspace(nbytes, dev)
    _check(_lib.attn_partial_pos(ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                 _ptr(v_scale), _ptr(seq_lens), _ptr(bounds), n_split, _ptr(q_pos), _ptr(k_pos),
                                 _ptr(out_partial), _ptr(lse_partial), _ptr(ws), nbytes, _stream()))
    return out_partial, lse_partial


@_on_tensor_device
def gqa_decode_attn_pos(q, k_cache, v_cache, seq_lens, split_bounds, q_pos, k_pos, k_scale=None, v_scale=None,
                        softmax_scale=None, scale_block=64, out=None, lse=None, workspace=None):
    """gqa_decode_attn with the causal rule taken from original positions (see attn_partial_pos)."""
    d, bounds, n_split = _prep(q, k_cache, v_cache, seq_lens, split_bounds, k_scale, v_scale, softmax_scale,
                               scale_block)
    _positions(q_pos, k_pos, d, q.device)
    dev = q.device
    out = _out(out, (d.B, d.Tq, d.Hq, d.dv), torch.bfloat16, dev, "out")
    lse = _out(lse, (d.B, d.Tq, d.Hq), torch.float32, dev, "lse")
    ws, ws_bytes = _ws_arg(workspace, gqa_decode_attn_workspace_size(d, n_split), dev)
    _check(_lib.gqa_decode_attn_pos(ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                    _ptr(v_scale), _ptr(seq_lens), _ptr(bounds), n_split, _ptr(q_pos), _ptr(k_pos),
                                    _ptr(out), _ptr(lse), _ptr(ws), ws_bytes, _stream()))
    return out, lse


@_on_tensor_device
def attn_partial_paged(q, k_pages, v_pages, seq_lens, split_bounds, block_table, causal_offset=NO_CAUSAL,
                       k_scale=None, v_scale=None, softmax_scale=None, scale_block=64, out_partial=None,
                       lse_partial=None):
    """attn_partial over a paged cache (pages [num_blocks,Hkv,block_len,d], block table
    int32 [B,max_blocks]; split bounds and seq_lens in logical tokens)."""
    d, pg, bounds, n_split = _prep_paged(q, k_pages, v_pages, seq_lens, split_bounds, block_table, k_scale, v_scale,
                                         softmax_scale, scale_block)
    dev = q.device
    out_partial = _out(out_partial, (n_split, d.B, d.Tq, d.Hq, d.dv), torch.float32, dev, "out_partial")
    lse_partial = _out(lse_partial, (n_split, d.B, d.Tq, d.Hq), torch.float32, dev, "lse_partial")
    nbytes = attn_partial_workspace_size(d, n_split)
    ws = _workspace(nbytes, dev)
    _check(_lib.attn_partial_paged(ctypes.byref(d), ctypes.byref(pg), _ptr(q), _ptr(k_pages), _ptr(v_pages),
                                   _ptr(k_scale), _ptr(v_scale), _ptr(seq_lens), _ptr(bounds), n_split, int(causal_offset),
                                   _ptr(out_partial), _ptr(lse_partial), _ptr(ws), nbytes, _stream()))
    return out_partial, lse_partial


@_on_tensor_device
def gqa_decode_attn_paged(q, k_pages, v_pages, seq_lens, split_bounds, block_table, causal_offset=NO_CAUSAL,
                          k_scale=None, v_scale=None, softmax_scale=None, scale_block=64, out=None, lse=None,
                          workspace=None):
    """gqa_decode_attn over a paged cache (see attn_partial_paged)."""
    d, pg, bounds, n_split = _prep_paged(q, k_pages, v_pages, seq_lens, split_bounds, block_table, k_scale, v_scale,
                                         softmax_scale, scale_block)
    dev = q.device
    out = _out(out, (d.B, d.Tq, d.Hq, d.dv), torch.bfloat16, dev, "out")
    lse = _out(lse, (d.B, d.Tq, d.Hq), torch.float32, dev, "lse")
    ws, ws_bytes = _ws_arg(workspace, gqa_decode_attn_workspace_size(d, n_split), dev)
    _check(_lib.gqa_decode_attn_paged(ctypes.byref(d), ctypes.byref(pg), _ptr(q), _ptr(k_pages), _ptr(v_pages),
                                      _ptr(k_scale), _ptr(v_scale), _ptr(seq_lens), _ptr(bounds), n_split,
                                      int(causal_offset), _ptr(out), _ptr(lse), _ptr(ws), ws_bytes, _stream()))
    return out, lse


@_on_tensor_device
def attn_ring_step(q, k_block, v_block, seq_lens, o_acc, lse_acc, causal_offset=NO_CAUSAL, first=False, k_scale=None,
                   v_scale=None, softmax_scale=None, scale_block=64):
    """One pass-KV ring step: attention of q over this step's KV block (its own buffer,
    [B,Hkv,S_blk,d]) merged into the running o_acc fp32 [B,Tq,Hq,dv] / lse_acc fp32
    [B,Tq,Hq] in place (written, not read, when first).  Returns (o_acc, lse_acc)."""
    _require_cuda(o_acc, lse_acc)
    _same_device(q.device, o_acc=o_acc, lse_acc=lse_acc)
    d, _, _ = _prep(q, k_block, v_block, seq_lens, None, k_scale, v_scale, softmax_scale, scale_block)
    for t, shape, name in ((o_acc, (d.B, d.Tq, d.Hq, d.dv), "o_acc"), (lse_acc, (d.B, d.Tq, d.Hq), "lse_acc")):
        if t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be contiguous float32 of shape {shape}")
    n = ctypes.c_size_t(0)
    _check(_lib.attn_ring_step_workspace_size(ctypes.byref(d), ctypes.byref(n)))
    ws = _workspace(int(n.value), q.device)
    _check(_lib.attn_ring_step(ctypes.byref(d), _ptr(q), _ptr(k_block), _ptr(v_block), _ptr(k_scale), _ptr(v_scale),
                               _ptr(seq_lens), int(causal_offset), 1 if first else 0, _ptr(o_acc), _ptr(lse_acc),
                               _ptr(ws), int(n.value), _stream()))
    return o_acc, lse_acc


@_on_tensor_device
def gqa_decode_attn_passq(q, k_shards, v_shards, shard_lens, k_scale=None, v_scale=None, softmax_scale=None,
                          scale_block=64, out=None, lse=None, workspace=None):
    """Pass-Q decode over the N = shard_lens.shape[0] ranks of a context-parallel group,
    emulated on this GPU: q bf16 [B,1,Hq,dk] (rank r owns requests [r*B/N, (r+1)*B/N));
    k_shards / v_shards [N*B,Hkv,S_loc,d] (row r*B+b: rank r's resident shard of request
    b); shard_lens int32 [N,B]; fp8 scales [N*B,Hkv,S_loc/scale_block].  Returns (out bf16
    [B,1,Hq,dv], lse fp32 [B,1,Hq])."""
    _require_cuda(q, k_shards, v_shards, shard_lens, k_scale, v_scale)
    _same_device(q.device, k_shards=k_shards, v_shards=v_shards, shard_lens=shard_lens, k_scale=k_scale,
                 v_scale=v_scale)
    if shard_lens.dtype != torch.int32 or not shard_lens.is_contiguous() or shard_lens.dim() != 2:
        raise ValueError("shard_lens must be contiguous int32 [n_ranks, B]")
    n_ranks, B = shard_lens.shape
    if k_shards.dim() != 4 or k_shards.shape[0] != n_ranks * B or v_shards.shape[0] != n_ranks * B:
        raise ValueError("k_shards / v_shards must be [n_ranks * B, Hkv, S_loc, d]")
    if q.dim() != 4 or q.shape[0] != B:
        raise ValueError("q must be [B, 1, Hq, dk] with B = shard_lens.shape[1]")
    # one shard row's description: the library steps through all n_ranks * B rows
    d = make_desc(q, k_shards[:B], v_shards[:B], softmax_scale, scale_block)
    if d.kv_dtype == SKV_KV_FP8_E4M3 and scale_block > 0:
        _check_scales((k_scale, v_scale), (n_ranks * B, d.Hkv, -(-d.S_max // scale_block)),
                      "[n_ranks * B, Hkv, ceil(S_loc / scale_block)]")
    dev = q.device
    out = _out(out, (d.B, d.Tq, d.Hq, d.dv), torch.bfloat16, dev, "out")
    lse = _out(lse, (d.B, d.Tq, d.Hq), torch.float32, dev, "lse")
    n = ctypes.c_size_t(0)
    _check(_lib.gqa_decode_attn_passq_workspace_size(ctypes.byref(d), n_ranks, ctypes.byref(n)))
    ws, ws_bytes = _ws_arg(workspace, int(n.value), dev)
    _check(_lib.gqa_decode_attn_passq(ctypes.byref(d), n_ranks, _ptr(q), _ptr(k_shards), _ptr(v_shards),
                                      _ptr(k_scale), _ptr(v_scale), _ptr(shard_lens), _ptr(out), _ptr(lse), _ptr(ws),
                                      ws_bytes, _stream()))
    return out, lse


def kernel_timing(enable):
    """Start (True: clears the record) or stop recording the attention kernels' own device time."""
    _check(_lib.splitkv_kernel_timing(1 if enable else 0))


def kernel_timing_read():
    """(total milliseconds, launches) of the attention kernels recorded since timing was enabled."""
    ms = ctypes.c_float(0.0)
    n = ctypes.c_int32(0)
    _check(_lib.splitkv_kernel_timing_read(ctypes.byref(ms), ctypes.byref(n)))
    return float(ms.value), int(n.value)


__all__ = [
    "kernel_timing",
    "kernel_timing_read",
    "attn_ring_step",
    "gqa_decode_attn_passq",
    "attn_partial",
    "attn_partial_paged",
    "gqa_decode_attn_paged",
    "attn_partial_pos",
    "attn_merge_lse",
    "gqa_decode_attn",
    "gqa_decode_attn_noalloc",
    "gqa_decode_attn_pos",
    "make_desc",
    "device_error",
    "last_error",
    "version",
    "SplitKVError",
    "SkvDesc",
    "LIB_PATH",
    "load_library",
    "EXPORTED_SYMBOLS",
    "NO_CAUSAL",
]
