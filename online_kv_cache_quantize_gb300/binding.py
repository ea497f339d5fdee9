"""ctypes binding of libtq (include/tq.h): the same entry-point names, argument
marshalling only. Every step of the hot path runs in the library's CUDA
kernels; PyTorch supplies device memory and streams.

The library is loaded on first use from this package directory. If it is
missing, every call raises: there is no CPU fallback.
"""

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libtq.so")
_lib = None

TQ_OK = 0
TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED = 1, 2
TQ_ERR_TIMEOUT = 6
TQ_ERR_WORKSPACE = 7
TQ_ROT_DENSE_QR, TQ_ROT_RHT = 0, 1
TQ_MSE, TQ_PROD, TQ_POLAR = 0, 1, 2
TQ_F32, TQ_BF16, TQ_F16 = 0, 1, 2

ROT_KINDS = {"dense": TQ_ROT_DENSE_QR, "rht": TQ_ROT_RHT}
MODES = {"mse": TQ_MSE, "prod": TQ_PROD, "polar": TQ_POLAR}


class TQError(RuntimeError):
    def __init__(self, status, where, message):
        super().__init__(f"{where}: {status_name(status)} ({message})")
        self.status = status


class tq_cache(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("bits", ctypes.c_int), ("d", ctypes.c_int), ("m", ctypes.c_int),
                ("rows", ctypes.c_int64), ("capacity", ctypes.c_int64),
                ("codes", ctypes.c_void_p), ("signs", ctypes.c_void_p),
                ("norm", ctypes.c_void_p), ("rnorm", ctypes.c_void_p), ("bits2", ctypes.c_int)]


class tq_quant_args(ctypes.Structure):
    _fields_ = [("cache", tq_cache), ("rot", ctypes.c_void_p), ("qjl", ctypes.c_void_p),
                ("x", ctypes.c_void_p), ("x_dtype", ctypes.c_int), ("x_stride", ctypes.c_int64),
                ("n", ctypes.c_int64), ("dst_slot", ctypes.c_void_p), ("append_pos", ctypes.c_void_p),
                ("heads", ctypes.c_int), ("slot0", ctypes.c_int64)]


class tq_decode_args(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("q_dtype", ctypes.c_int),
                ("batch", ctypes.c_int), ("hq", ctypes.c_int), ("hkv", ctypes.c_int), ("d", ctypes.c_int),
                ("seq_lens", ctypes.c_void_p), ("max_seq_len", ctypes.c_int),
                ("gqa_map", ctypes.c_void_p), ("rot", ctypes.c_void_p), ("qjl", ctypes.c_void_p),
                ("k", tq_cache), ("v", tq_cache), ("scale", ctypes.c_float), ("n_splits", ctypes.c_int),
                ("out", ctypes.c_void_p), ("out_dtype", ctypes.c_int), ("logits", ctypes.c_void_p),
                ("scan_begin", ctypes.c_void_p), ("scan_end", ctypes.c_void_p)]


class tq_step_args(ctypes.Structure):
    _fields_ = [("attn", tq_decode_args), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("new_dtype", ctypes.c_int), ("append_pos", ctypes.c_void_p)]


class tq_prefill_args(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("q_dtype", ctypes.c_int),
                ("batch", ctypes.c_int), ("chunk", ctypes.c_int), ("hq", ctypes.c_int), ("hkv", ctypes.c_int),
                ("d", ctypes.c_int), ("q_start", ctypes.c_void_p), ("max_context", ctypes.c_int),
                ("gqa_map", ctypes.c_void_p), ("rot", ctypes.c_void_p), ("qjl", ctypes.c_void_p), ("k", tq_cache), ("v", tq_cache),
                ("scale", ctypes.c_float), ("n_splits", ctypes.c_int), ("out", ctypes.c_void_p),
                ("out_dtype", ctypes.c_int), ("scan_begin", ctypes.c_void_p), ("scan_end", ctypes.c_void_p)]


class tq_topk_args(ctypes.Structure):
    _fields_ = [("queries", ctypes.c_void_p), ("nq", ctypes.c_int), ("d", ctypes.c_int),
                ("rot", ctypes.c_void_p), ("qjl", ctypes.c_void_p), ("db", tq_cache),
                ("n_db", ctypes.c_int64), ("k", ctypes.c_int), ("ids", ctypes.c_void_p),
                ("scores", ctypes.c_void_p)]


_STATUS = ctypes.c_int
_SIGS = {
    "tq_status_string": (ctypes.c_char_p, [_STATUS]),
    "tq_last_error": (ctypes.c_char_p, []),
    "tq_abi_struct_size": (ctypes.c_size_t, [ctypes.c_char_p]),
    "tq_random_stream": (_STATUS, [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p]),
    "tq_make_rotation": (_STATUS, [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)]),
    "tq_rotation_get": (_STATUS, [ctypes.c_void_p, ctypes.c_void_p]),
    "tq_rotation_info": (_STATUS, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "tq_rotation_to_device": (_STATUS, [ctypes.c_void_p]),
    "tq_free_rotation": (_STATUS, [ctypes.c_void_p]),
    "tq_make_qjl": (_STATUS, [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)]),
    "tq_qjl_get": (_STATUS, [ctypes.c_void_p, ctypes.c_void_p]),
    "tq_qjl_to_device": (_STATUS, [ctypes.c_void_p]),
    "tq_free_qjl": (_STATUS, [ctypes.c_void_p]),
    "tq_codebook": (_STATUS, [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "tq_code_bytes": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "tq_code_bytes2": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "tq_sign_bytes": (ctypes.c_int, [ctypes.c_int]),
    "tq_polar_code_bytes": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "tq_polar_codebook": (_STATUS, [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "tq_quantize_kv": (_STATUS, [ctypes.POINTER(tq_quant_args), ctypes.c_void_p]),
    "tq_attn_decode_workspace": (ctypes.c_size_t, [ctypes.POINTER(tq_decode_args)]),
    "tq_attn_decode": (_STATUS, [ctypes.POINTER(tq_decode_args), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "tq_attn_prefill_workspace": (ctypes.c_size_t, [ctypes.POINTER(tq_prefill_args)]),
    "tq_attn_prefill": (_STATUS, [ctypes.POINTER(tq_prefill_args), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "tq_attn_decode_static": (_STATUS, [ctypes.POINTER(tq_decode_args), ctypes.c_void_p]),
    "tq_score_topk_workspace": (ctypes.c_size_t, [ctypes.POINTER(tq_topk_args)]),
    "tq_score_topk": (_STATUS, [ctypes.POINTER(tq_topk_args), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "tq_decode_step_workspace": (ctypes.c_size_t, [ctypes.POINTER(tq_step_args)]),
    "tq_decode_step": (_STATUS, [ctypes.POINTER(tq_step_args), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "tq_topk_force_simt": (ctypes.c_int, [ctypes.c_int]),
    "tq_quantize_force_mma_sync": (ctypes.c_int, [ctypes.c_int]),
    "tq_prefill_force_mma_sync": (ctypes.c_int, [ctypes.c_int]),
    "tq_device_errors": (_STATUS, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
    "tq_selftest_bounded_wait": (_STATUS, [ctypes.c_uint32, ctypes.c_void_p]),
    "tq_selftest_umma_gemm": (_STATUS, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p]),
    "tq_selftest_umma_gemm_tmem_a": (_STATUS, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p]),
}

EXPORTED = tuple(_SIGS)


def lib_path():
    return _LIB_PATH


def load():
    """Load libtq.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"libtq.so not built at {_LIB_PATH}; run online_kv_cache_quantize_gb300.build")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    for name, cls in (("tq_cache", tq_cache), ("tq_quant_args", tq_quant_args),
                      ("tq_decode_args", tq_decode_args), ("tq_topk_args", tq_topk_args),
                      ("tq_step_args", tq_step_args), ("tq_prefill_args", tq_prefill_args)):
        if lib.tq_abi_struct_size(name.encode()) != ctypes.sizeof(cls):
            raise RuntimeError(f"struct {name} layout differs between libtq.so and the binding")
    _lib = lib
    return lib


def status_name(s):
    return load().tq_status_string(s).decode()


def _check(status, where):
    if status != TQ_OK:
        raise TQError(status, where, load().tq_last_error().decode())


# ---------------------------------------------------------------- set-up ---
def tq_random_stream(seed, count, start=0):
    out = np.empty(count, dtype=np.uint64)
    _check(load().tq_random_stream(seed, start, count, out.ctypes.data), "tq_random_stream")
    return out


class Rotation:
    """Owns a tq_rotation handle."""

    def __init__(self, handle, d, kind):
        self.handle, self.d, self.kind = handle, d, kind

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.tq_free_rotation(self.handle)
            self.handle = None


class QJL:
    """Owns a tq_qjl handle."""

    def __init__(self, handle, m, d):
        self.handle, self.m, self.d = handle, m, d

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.tq_free_qjl(self.handle)
            self.handle = None


def tq_make_rotation(seed, d, kind="dense"):
    h = ctypes.c_void_p()
    k = ROT_KINDS.get(kind, kind)
    _check(load().tq_make_rotation(seed, d, k, ctypes.byref(h)), "tq_make_rotation")
    return Rotation(h.value, d, k)


def tq_rotation_get(rot):
    out = np.empty((rot.d, rot.d), dtype=np.float64)
    _check(load().tq_rotation_get(rot.handle, out.ctypes.data), "tq_rotation_get")
    return out


def tq_rotation_to_device(rot):
    _check(load().tq_rotation_to_device(rot.handle), "tq_rotation_to_device")
    return rot


def tq_make_qjl(seed, m, d):
    h = ctypes.c_void_p()
    _check(load().tq_make_qjl(seed, m, d, ctypes.byref(h)), "tq_make_qjl")
    return QJL(h.value, m, d)


def tq_qjl_get(qjl):
    out = np.empty((qjl.m, qjl.d), dtype=np.float64)
    _check(load().tq_qjl_get(qjl.handle, out.ctypes.data), "tq_qjl_get")
    return out


def tq_qjl_to_device(qjl):
    _check(load().tq_qjl_to_device(qjl.handle), "tq_qjl_to_device")
    return qjl


def tq_codebook(d, bits):
    c = np.empty(1 << bits, dtype=np.float64)
    t = np.empty((1 << bits) - 1, dtype=np.float64)
    _check(load().tq_codebook(d, bits, c.ctypes.data, t.ctypes.data), "tq_codebook")
    return c, t


def tq_code_bytes(d, code_bits):
    return load().tq_code_bytes(d, code_bits)


def tq_sign_bytes(m):
    return load().tq_sign_bytes(m)


def tq_polar_code_bytes(d, bits1, bits2):
    return load().tq_polar_code_bytes(d, bits1, bits2)


def tq_polar_codebook(level, bits):
    c = np.empty(1 << bits, dtype=np.float64)
    t = np.empty((1 << bits) - 1, dtype=np.float64)
    _check(load().tq_polar_codebook(level, bits, c.ctypes.data, t.ctypes.data), "tq_polar_codebook")
    return c, t


# ------------------------------------------------------- cache planes ---
class Cache:
    """Device planes of a packed cache (torch tensors owned by this object)."""

    def __init__(self, mode, bits, d, rows, capacity, m=None, device="cuda", bits2=None):
        """bits2: the second channel group's bits of a fractional-rate cache
        (coordinates with i % 16 >= 8), None for one width; for a PolarQuant
        cache ("polar") the bits of the angles above level 1 (required)."""
        import torch

        self.mode = MODES.get(mode, mode)
        self.bits, self.d, self.rows, self.capacity = bits, d, rows, capacity
        if self.mode == TQ_POLAR:
            if not bits2:
                raise ValueError("a PolarQuant cache needs bits2 (the bits of the angles above level 1)")
            self.bits2 = bits2
        else:
            self.bits2 = bits2 if bits2 and bits2 != bits else None
        self.m = (m if m is not None else d) if self.mode == TQ_PROD else 0
        cb = bits - 1 if self.mode == TQ_PROD else bits
        self.code_bits = cb
        n = rows * capacity
        if self.mode == TQ_POLAR:
            self.code_stride = tq_polar_code_bytes(d, bits, bits2)
        elif self.bits2 is None:
            self.code_stride = tq_code_bytes(d, cb)
        else:
            self.code_stride = load().tq_code_bytes2(d, cb, self.bits2 - 1 if self.mode == TQ_PROD else self.bits2)
        self.codes = torch.zeros((n, self.code_stride), dtype=torch.uint8, device=device)
        self.norm = torch.zeros(n, dtype=torch.int16, device=device)
        if self.mode == TQ_PROD:
            self.sign_stride = tq_sign_bytes(self.m)
            self.signs = torch.zeros((n, self.sign_stride), dtype=torch.uint8, device=device)
            self.rnorm = torch.zeros(n, dtype=torch.int16, device=device)
        else:
            self.sign_stride = 0
            self.signs = None
            self.rnorm = None

    def struct(self):
        return tq_cache(self.mode, self.bits, self.d, self.m, self.rows, self.capacity,
                        self.codes.data_ptr(), self.signs.data_ptr() if self.signs is not None else None,
                        self.norm.data_ptr(), self.rnorm.data_ptr() if self.rnorm is not None else None,
                        self.bits2 or 0)

    def bytes_per_slot(self):
        return self.code_stride + 2 + (self.sign_stride + 2 if self.mode == TQ_PROD else 0)


def _dtype_code(t):
    import torch

    return {torch.float32: TQ_F32, torch.bfloat16: TQ_BF16, torch.float16: TQ_F16}[t.dtype]


def _stream_ptr(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


# ------------------------------------------------------------- hot path ---
def tq_quantize_kv(cache, rot, x, qjl=None, slot0=0, dst_slot=None, append_pos=None, heads=1, stream=None):
    """Quantize rows of x (device [n, >=d], f32 or bf16) into `cache`."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D tensor with unit inner stride")
    a = tq_quant_args()
    a.cache = cache.struct()
    a.rot = rot.handle
    a.qjl = qjl.handle if qjl is not None else None
    a.x = x.data_ptr()
    a.x_dtype = _dtype_code(x)
    a.x_stride = x.stride(0)
    a.n = x.shape[0]
    a.dst_slot = dst_slot.data_ptr() if dst_slot is not None else None
    a.append_pos = append_pos.data_ptr() if append_pos is not None else None
    a.heads = heads
    a.slot0 = slot0
    _check(load().tq_quantize_kv(ctypes.byref(a), _stream_ptr(stream)), "tq_quantize_kv")


def _decode_struct(q, kcache, vcache, seq_lens, max_seq_len, rot, qjl, out, scale=0.0, n_splits=0,
                   gqa_map=None, logits=None):
    b, hq, d = q.shape
    a = tq_decode_args()
    a.q = q.data_ptr()
    a.q_dtype = _dtype_code(q)
    a.batch, a.hq, a.hkv, a.d = b, hq, kcache.rows // b, d
    a.seq_lens = seq_lens.data_ptr()
    a.max_seq_len = max_seq_len
    keep = None
    if gqa_map is not None:
        keep = np.ascontiguousarray(gqa_map, dtype=np.int32)
        a.gqa_map = keep.ctypes.data
    a.rot = rot.handle
    a.qjl = qjl.handle if qjl is not None else None
    a.k = kcache.struct()
    a.v = vcache.struct()
    a.scale = scale
    a.n_splits = n_splits
    a.out = out.data_ptr()
    a.out_dtype = _dtype_code(out)
    a.logits = logits.data_ptr() if logits is not None else None
    return a, keep


def tq_attn_decode_workspace(q, kcache, vcache, seq_lens, max_seq_len, rot, qjl, out, **kw):
    a, _keep = _decode_struct(q, kcache, vcache, seq_lens, max_seq_len, rot, qjl, out, **kw)
    return load().tq_attn_decode_workspace(ctypes.byref(a))


def tq_attn_decode(q, kcache, vcache, seq_lens, max_seq_len, rot, qjl, out, workspace, stream=None, **kw):
    """Decode attention over the packed caches; writes `out` (and `logits` if given)."""
    a, _keep = _decode_struct(q, kcache, vcache, seq_lens, max_seq_len, rot, qjl, out, **kw)
    _check(load().tq_attn_decode(ctypes.byref(a), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream)), "tq_attn_decode")


def _prefill_struct(q, kcache, vcache, q_start, max_context, rot, qjl, out, scale=0.0, n_splits=0, gqa_map=None,
                    scan_events=None):
    b, c, hq, d = q.shape
    a = tq_prefill_args()
    keep = None
    if gqa_map is not None:
        keep = np.ascontiguousarray(gqa_map, dtype=np.int32)
        a.gqa_map = keep.ctypes.data
    a.q = q.data_ptr()
    a.q_dtype = _dtype_code(q)
    a.batch, a.chunk, a.hq, a.hkv, a.d = b, c, hq, kcache.rows // b, d
    a.q_start = q_start.data_ptr()
    a.max_context = max_context
    a.rot = rot.handle
    a.qjl = qjl.handle if qjl is not None else None
    a.k = kcache.struct()
    a.v = vcache.struct()
    a.scale = scale
    a.n_splits = n_splits
    a.out = out.data_ptr()
    a.out_dtype = _dtype_code(out)
    if scan_events is not None:  # (begin, end) torch.cuda.Event pair, recorded around the scan kernel
        a.scan_begin = scan_events[0].cuda_event
        a.scan_end = scan_events[1].cuda_event
    return a, keep


def tq_attn_prefill_workspace(q, kcache, vcache, q_start, max_context, rot, qjl, out, **kw):
    a, _keep = _prefill_struct(q, kcache, vcache, q_start, max_context, rot, qjl, out, **kw)
    return load().tq_attn_prefill_workspace(ctypes.byref(a))


def tq_attn_prefill(q, kcache, vcache, q_start, max_context, rot, qjl, out, workspace, stream=None, **kw):
    """Chunked-prefill attention: q [batch][chunk][hq][d], the chunk of each
    sequence starting at position q_start[b] (device int32) and already
    quantized into the caches; writes out [batch][chunk][hq][d]."""
    a, _keep = _prefill_struct(q, kcache, vcache, q_start, max_context, rot, qjl, out, **kw)
    _check(load().tq_attn_prefill(ctypes.byref(a), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                  _stream_ptr(stream)), "tq_attn_prefill")


def tq_attn_decode_static(q, kcache, vcache, seq_lens, max_seq_len, rot, qjl, out, stream=None, **kw):
    """tq_attn_decode without a workspace: for callers that may not allocate
    device memory; its scratch is an array inside the library (see tq.h)."""
    a, _keep = _decode_struct(q, kcache, vcache, seq_lens, max_seq_len, rot, qjl, out, **kw)
    _check(load().tq_attn_decode_static(ctypes.byref(a), _stream_ptr(stream)), "tq_attn_decode_static")


def _step_struct(q, kcache, vcache, seq_lens, max_seq_len, rot, qjl, out, k_new, v_new, append_pos, **kw):
    attn, keep = _decode_struct(q, kcache, vcache, seq_lens, max_seq_len, rot, qjl, out, **kw)
    a = tq_step_args()
    a.attn = attn
    a.k_new = k_new.data_ptr()
    a.v_new = v_new.data_ptr()
    if k_new.dtype != v_new.dtype:
        raise ValueError("k_new and v_new must have the same dtype")
    a.new_dtype = _dtype_code(k_new)
    a.append_pos = append_pos.data_ptr()
    return a, keep


def tq_decode_step_workspace(q, kcache, vcache, seq_lens, max_seq_len, rot, qjl, out, k_new, v_new, append_pos, **kw):
    a, _keep = _step_struct(q, kcache, vcache, seq_lens, max_seq_len, rot, qjl, out, k_new, v_new, append_pos, **kw)
    return load().tq_decode_step_workspace(ctypes.byref(a))


def tq_decode_step(q, kcache, vcache, seq_lens, max_seq_len, rot, qjl, out, k_new, v_new, append_pos, workspace,
                   stream=None, **kw):
    """Append the new token's K and V (rows b*hkv + h of k_new / v_new at slot
    append_pos[b]) and run decode attention, in one call."""
    a, _keep = _step_struct(q, kcache, vcache, seq_lens, max_seq_len, rot, qjl, out, k_new, v_new, append_pos, **kw)
    _check(load().tq_decode_step(ctypes.byref(a), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream)), "tq_decode_step")


TQ_DEVERR_SCAN_WAIT = 1
TQ_DEVERR_SELFTEST_WAIT = 2
TQ_DEVERR_QUANT_WAIT = 4


def tq_device_errors(reset=False):
    """(status, flags) of the current device's error word; synchronises the device."""
    v = ctypes.c_uint32(0)
    st = load().tq_device_errors(ctypes.byref(v), 1 if reset else 0)
    if st not in (TQ_OK, TQ_ERR_TIMEOUT):
        _check(st, "tq_device_errors")
    return st, v.value


def tq_selftest_bounded_wait(limit_us, stream=None):
    """One warp waits on an mbarrier nothing arrives on, at most limit_us."""
    _check(load().tq_selftest_bounded_wait(limit_us, _stream_ptr(stream)), "tq_selftest_bounded_wait")


def tq_selftest_umma_gemm(a, b, d, stream=None, a_in_tmem=False):
    """d[128][n] = a[128][k] @ b[n][k]^T on the tcgen05 tensor-core path (fp16 in, fp32 out);
    a_in_tmem: the MMA reads A from tensor memory instead of shared memory."""
    n, k = b.shape
    fn = load().tq_selftest_umma_gemm_tmem_a if a_in_tmem else load().tq_selftest_umma_gemm
    _check(fn(a.data_ptr(), b.data_ptr(), d.data_ptr(), n, k, _stream_ptr(stream)), "tq_selftest_umma_gemm")


def _topk_struct(queries, db, n_db, rot, qjl, k, ids, scores):
    a = tq_topk_args()
    a.queries = queries.data_ptr()
    a.nq, a.d = queries.shape
    a.rot = rot.handle
    a.qjl = qjl.handle if qjl is not None else None
    a.db = db.struct()
    a.n_db = n_db
    a.k = k
    a.ids = ids.data_ptr()
    a.scores = scores.data_ptr()
    return a


def tq_score_topk_workspace(queries, db, n_db, rot, qjl, k, ids, scores):
    a = _topk_struct(queries, db, n_db, rot, qjl, k, ids, scores)
    return load().tq_score_topk_workspace(ctypes.byref(a))


def tq_score_topk(queries, db, n_db, rot, qjl, k, ids, scores, workspace, stream=None):
    a = _topk_struct(queries, db, n_db, rot, qjl, k, ids, scores)
    _check(load().tq_score_topk(ctypes.byref(a), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                _stream_ptr(stream)), "tq_score_topk")


def workspace(nbytes, device="cuda"):
    """A 256-byte aligned device byte buffer (torch allocations are)."""
    import torch

    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


class QuantizedKVCache:
    """One attention layer's packed KV cache with the decode loop's calls:
    `prefill` quantizes a context into it, `prefill_chunk` appends a chunk of
    tokens per batch row and attends with the chunk's queries (causal), and
    `step` appends one token per batch row and attends (the write-ups'
    "quantize on every cache update, then attend"; tq_quantize_kv,
    tq_attn_prefill and tq_decode_step). Keys are PROD (k_bits,
    QJL signs), values MSE (v_bits); both share one rotation. The per-row
    lengths live on the device; this class only keeps the handles, the
    planes and a workspace, and forms the calls' arguments."""

    def __init__(self, batch, hq, hkv, capacity, d=128, k_bits=3, v_bits=3, rotation="rht", rot_seed=1, qjl_seed=2,
                 device="cuda", k_bits2=None, v_bits2=None):
        import torch

        if hq % hkv:
            raise ValueError("hq must be a multiple of hkv")
        self.batch, self.hq, self.hkv, self.capacity, self.d = batch, hq, hkv, capacity, d
        self.rot = tq_rotation_to_device(tq_make_rotation(rot_seed, d, rotation))
        self.qjl = tq_qjl_to_device(tq_make_qjl(qjl_seed, d, d))
        self.k = Cache("prod", k_bits, d, rows=batch * hkv, capacity=capacity, device=device, bits2=k_bits2)
        self.v = Cache("mse", v_bits, d, rows=batch * hkv, capacity=capacity, device=device, bits2=v_bits2)
        self.lengths = torch.zeros(batch, dtype=torch.int32, device=device)
        self._host_lengths = [0] * batch  # the same lengths, for the launch plans
        self._ws = None

    def prefill(self, k, v, lengths):
        """k, v: device [batch, hkv, T, d] (f32 or bf16), T <= capacity; row b
        holds lengths[b] valid tokens (a host sequence of ints)."""
        import torch

        b, h, t, d = k.shape
        if (b, h, d) != (self.batch, self.hkv, self.d) or tuple(v.shape) != tuple(k.shape) or t > self.capacity:
            raise ValueError("k and v must be [batch, hkv, T <= capacity, d]")
        lens = [int(x) for x in lengths]
        if len(lens) != b or min(lens) < 0 or max(lens) > t:
            raise ValueError("lengths must give 0 <= length <= T per batch row")
        # slot of token j of (b, h): (b * hkv + h) * capacity + j; tokens past a row's length are skipped
        j = torch.arange(t, device=k.device, dtype=torch.int64)
        rows = torch.arange(b * h, device=k.device, dtype=torch.int64)
        slots = rows[:, None] * self.capacity + j[None, :]
        valid = j[None, :] < torch.tensor(lens, device=k.device, dtype=torch.int64).repeat_interleave(h)[:, None]
        slots = torch.where(valid, slots, torch.full_like(slots, -1)).reshape(-1).contiguous()
        tq_quantize_kv(self.k, self.rot, k.reshape(-1, d), qjl=self.qjl, dst_slot=slots)
        tq_quantize_kv(self.v, self.rot, v.reshape(-1, d), dst_slot=slots)
        self.lengths.copy_(torch.tensor(lens, dtype=torch.int32))
        self._host_lengths = lens

    def prefill_chunk(self, q, k, v, out=None, stream=None):
        """Appends a chunk of C tokens to every batch row (k, v: device
        [batch, hkv, C, d]) at the row's current length, then attends with the
        chunk's queries (device [batch, C, hq, d]; query i sees the row's
        tokens up to and including chunk token i). Returns out
        ([batch, C, hq, d], fp32 unless given)."""
        import torch

        b, h, c, d = k.shape
        if (b, h, d) != (self.batch, self.hkv, self.d) or tuple(v.shape) != tuple(k.shape):
            raise ValueError("k and v must be [batch, hkv, C, d]")
        if tuple(q.shape) != (b, c, self.hq, d):
            raise ValueError("q must be [batch, C, hq, d]")
        max_context = max(self._host_lengths) + c
        if max_context > self.capacity:
            raise ValueError("the chunk does not fit the capacity")
        if out is None:
            out = torch.empty((b, c, self.hq, d), dtype=torch.float32, device=q.device)
        # slot of chunk token j of (b, h): (b * hkv + h) * capacity + lengths[b] + j
        j = torch.arange(c, device=k.device, dtype=torch.int64)
        rows = torch.arange(b * h, device=k.device, dtype=torch.int64)
        start = self.lengths.to(torch.int64).repeat_interleave(h)
        slots = (rows[:, None] * self.capacity + start[:, None] + j[None, :]).reshape(-1).contiguous()
        tq_quantize_kv(self.k, self.rot, k.reshape(-1, d), qjl=self.qjl, dst_slot=slots, stream=stream)
        tq_quantize_kv(self.v, self.rot, v.reshape(-1, d), dst_slot=slots, stream=stream)
        need = tq_attn_prefill_workspace(q, self.k, self.v, self.lengths, max_context, self.rot, self.qjl, out)
        if self._ws is None or self._ws.numel() < need:
            self._ws = workspace(need, device=q.device)
        tq_attn_prefill(q, self.k, self.v, self.lengths, max_context, self.rot, self.qjl, out, self._ws,
                        stream=stream)
        self.lengths = self.lengths + c
        self._host_lengths = [x + c for x in self._host_lengths]
        return out

    def step(self, q, k_new, v_new, out=None, stream=None):
        """Appends k_new / v_new (device [batch, hkv, d]) at each row's current
        length and attends with q (device [batch, hq, d]); returns out
        ([batch, hq, d], fp32 unless given). The caller keeps every length
        below the capacity."""
        import torch

        if out is None:
            out = torch.empty((self.batch, self.hq, self.d), dtype=torch.float32, device=q.device)
        kn = k_new.reshape(self.batch * self.hkv, self.d)
        vn = v_new.reshape(self.batch * self.hkv, self.d)
        new_lens = self.lengths + 1
        need = tq_decode_step_workspace(q, self.k, self.v, new_lens, self.capacity, self.rot, self.qjl, out, kn, vn,
                                        self.lengths)
        if self._ws is None or self._ws.numel() < need:
            self._ws = workspace(need, device=q.device)
        tq_decode_step(q, self.k, self.v, new_lens, self.capacity, self.rot, self.qjl, out, kn, vn, self.lengths,
                       self._ws, stream=stream)
        self.lengths = new_lens
        self._host_lengths = [x + 1 for x in self._host_lengths]
        return out
