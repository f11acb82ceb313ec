"""Thin ctypes binding over ``libint8kv.so`` (the C ABI of include/int8kv.h).

Only argument marshalling happens here: torch tensors are checked for device,
dtype and contiguity and turned into raw pointers; every step of the
computation runs in the library's CUDA kernels.  There is no fallback: when
the library is missing or a call fails, an exception is raised.

Function names follow the C ABI.  ``KVPool`` is a convenience owner of the
device regions (allocated with torch, which only provides memory).
"""

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libint8kv.so")

K8V8, K8V16, K16V8, K8V4, Q4_0 = 0, 1, 2, 3, 4
VARIANTS = {"k8v8": K8V8, "k8v16": K8V16, "k16v8": K16V8, "k8v4": K8V4, "q4_0": Q4_0}
REGION_K_STORE, REGION_V_STORE, REGION_K_SCALES, REGION_V_SCALES = 0, 1, 2, 3
DEVERR_PAGE_ID, DEVERR_LENGTH, DEVERR_TIMEOUT = 1, 2, 4
ERR_FORMAT = -9
DECODE_AUTO, DECODE_WARP_MMA, DECODE_SIMT = 0, 1, 3

_c_int, _c_size, _vp, _c_float = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
_SIGS = {
    "int8kv_status_string": (ctypes.c_char_p, [_c_int]),
    "int8kv_pool_region_bytes": (_c_int, [_c_int] * 8 + [ctypes.POINTER(_c_size)]),
    "kv_pool_create": (_c_int, [ctypes.POINTER(_vp)] + [_c_int] * 7 + [_vp] * 5),
    "kv_pool_destroy": (None, [_vp]),
    "kv_quant_append": (_c_int, [_vp, _c_int, _vp, _vp, _c_int, _c_int, _vp, _vp, _c_int, _vp]),
    "attn_decode_n_splits": (_c_int, [_vp, _c_int, _c_int]),
    "attn_decode_workspace_bytes": (_c_int, [_c_int] * 5 + [ctypes.POINTER(_c_size)]),
    "attn_decode_int8": (_c_int, [_vp, _c_int, _vp, _c_int, _c_int, _vp, _vp, _c_int, _c_int,
                                  _c_float, _c_int, _vp, _vp, _c_size, _vp]),
    "kv_pool_read_device_error": (_c_int, [_vp, ctypes.POINTER(ctypes.c_int32), _vp]),
    "attn_decode_append_int8": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _c_int, _c_int, _vp, _vp,
                                         _c_int, _c_int, _c_float, _c_int, _vp, _vp, _c_size,
                                         _vp]),
    "attn_decode_multi_int8": (_c_int, [_vp, _c_int, _vp, _c_int, _c_int, _c_int, _vp, _vp,
                                        _c_int, _c_float, _c_int, _vp, _vp, _c_size, _vp]),
    "attn_prefill_n_splits": (_c_int, [_vp, _c_int, _c_int, _c_int]),
    "attn_prefill_workspace_bytes": (_c_int, [_c_int] * 5 + [ctypes.POINTER(_c_size)]),
    "attn_prefill_chunk_int8": (_c_int, [_vp, _c_int, _vp, _c_int, _c_int, _c_int, _vp, _c_int,
                                         _c_float, _c_int, _vp, _vp, _c_size, _vp]),
    "attn_decode_int8_noalloc": (_c_int, [_vp, _c_int, _vp, _c_int, _c_int, _vp, _vp, _c_int,
                                          _c_int, _c_float, _c_int, _vp, _vp]),
    "kv_pool_set_decode_kernel": (_c_int, [_vp, _c_int]),
    "kv_pool_image_bytes": (_c_int, [_vp, _c_int, _vp, ctypes.POINTER(_c_size)]),
    "kv_pool_test_expire_waits": (_c_int, [_vp, ctypes.c_uint32]),
    "kv_pool_save": (_c_int, [_vp, _c_int, _vp, _vp, _c_int, _vp, _c_size, _vp, _c_size, _vp]),
    "kv_pool_load": (_c_int, [_vp, _vp, _c_size, _c_int, _vp, _c_int, _vp, _c_size, _vp, _vp]),
}

_lib = None


class Int8KVError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_name(status)} ({status})")


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "int8_kv_cache_02_gb300.build.build() (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_name(status):
    return lib().int8kv_status_string(status).decode()


def int8kv_status_string(status):
    return status_name(status)


def _check(status, where):
    if status != 0:
        raise Int8KVError(status, where)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t, dtype, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def int8kv_pool_region_bytes(n_layers, n_kv_heads, head_dim, group_size, page_size, n_pages,
                             variant, region):
    out = _c_size(0)
    _check(lib().int8kv_pool_region_bytes(n_layers, n_kv_heads, head_dim, group_size, page_size,
                                          n_pages, variant, region, ctypes.byref(out)),
           "int8kv_pool_region_bytes")
    return out.value


def kv_pool_create(n_layers, n_kv_heads, head_dim, group_size, page_size, n_pages, variant,
                   k_store, v_store, k_scales, v_scales, dev_error):
    """Raw descriptor over caller tensors (any dtype; only the pointers are used)."""
    h = ctypes.c_void_p()
    ptr = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    _check(lib().kv_pool_create(ctypes.byref(h), n_layers, n_kv_heads, head_dim, group_size,
                                page_size, n_pages, variant, ptr(k_store), ptr(v_store),
                                ptr(k_scales), ptr(v_scales), ptr(dev_error)), "kv_pool_create")
    return h


def kv_pool_destroy(handle):
    lib().kv_pool_destroy(handle)


def kv_quant_append(pool, layer, k_new, v_new, seq_pos, page_table, stream=None):
    """k_new, v_new: fp16 [n_seqs][n_new][Hkv][D]; seq_pos int32 [n_seqs];
    page_table int32 [n_seqs][max_pages]."""
    n_seqs, n_new = k_new.shape[0], k_new.shape[1]
    _check(lib().kv_quant_append(pool.handle, layer, _dev(k_new, torch.float16, "k_new"),
                                 _dev(v_new, torch.float16, "v_new"), n_seqs, n_new,
                                 _dev(seq_pos, torch.int32, "seq_pos"),
                                 _dev(page_table, torch.int32, "page_table"),
                                 page_table.shape[1], _stream(stream)), "kv_quant_append")


def attn_decode_n_splits(pool, batch, max_ctx):
    n = lib().attn_decode_n_splits(pool.handle, batch, max_ctx)
    if n < 0:
        raise Int8KVError(n, "attn_decode_n_splits")
    return n


def attn_decode_workspace_bytes(batch, n_heads, n_kv_heads, head_dim, n_splits):
    out = _c_size(0)
    _check(lib().attn_decode_workspace_bytes(batch, n_heads, n_kv_heads, head_dim, n_splits,
                                             ctypes.byref(out)), "attn_decode_workspace_bytes")
    return out.value


def attn_decode_int8(pool, layer, q, seq_lens, page_table, out, workspace=None, window=0,
                     softmax_scale=0.0, n_splits=0, stream=None):
    """q fp16 [B][H][D]; seq_lens int32 [B]; page_table int32 [B][max_pages];
    out fp32 [B][H][D]; workspace uint8 tensor (any contents) or None."""
    B, H = q.shape[0], q.shape[1]
    ws = _dev(workspace, torch.uint8, "workspace") if workspace is not None else None
    nbytes = workspace.numel() if workspace is not None else 0
    _check(lib().attn_decode_int8(pool.handle, layer, _dev(q, torch.float16, "q"), B, H,
                                  _dev(seq_lens, torch.int32, "seq_lens"),
                                  _dev(page_table, torch.int32, "page_table"),
                                  page_table.shape[1], window, float(softmax_scale), n_splits,
                                  _dev(out, torch.float32, "out"), ws, nbytes, _stream(stream)),
           "attn_decode_int8")


def attn_decode_int8_noalloc(pool, layer, q, seq_lens, page_table, out, window=0,
                             softmax_scale=0.0, n_splits=0, stream=None):
    """attn_decode_int8 without a workspace: the partials use the library's own
    fixed scratch (for callers that cannot allocate device memory)."""
    B, H = q.shape[0], q.shape[1]
    _check(lib().attn_decode_int8_noalloc(pool.handle, layer, _dev(q, torch.float16, "q"), B, H,
                                          _dev(seq_lens, torch.int32, "seq_lens"),
                                          _dev(page_table, torch.int32, "page_table"),
                                          page_table.shape[1], window, float(softmax_scale),
                                          n_splits, _dev(out, torch.float32, "out"),
                                          _stream(stream)), "attn_decode_int8_noalloc")


def attn_decode_append_int8(pool, layer, q, k_new, v_new, seq_lens, page_table, out,
                            workspace=None, window=0, softmax_scale=0.0, n_splits=0, stream=None):
    """Append k_new, v_new (fp16 [B][Hkv][D]) at position seq_lens[b] - 1, then decode."""
    B, H = q.shape[0], q.shape[1]
    ws = _dev(workspace, torch.uint8, "workspace") if workspace is not None else None
    nbytes = workspace.numel() if workspace is not None else 0
    _check(lib().attn_decode_append_int8(pool.handle, layer, _dev(q, torch.float16, "q"),
                                         _dev(k_new, torch.float16, "k_new"),
                                         _dev(v_new, torch.float16, "v_new"), B, H,
                                         _dev(seq_lens, torch.int32, "seq_lens"),
                                         _dev(page_table, torch.int32, "page_table"),
                                         page_table.shape[1], window, float(softmax_scale),
                                         n_splits, _dev(out, torch.float32, "out"), ws, nbytes,
                                         _stream(stream)), "attn_decode_append_int8")


def attn_decode_multi_int8(pool, layer, q, seq_lens, page_table, out, workspace=None,
                           softmax_scale=0.0, n_splits=0, stream=None):
    """Decode of a window of queries per sequence, causal within the window.

    q: fp16 [B][q_len][H][D]; query i of sequence b sits at position
    seq_lens[b] - q_len + i.  out: fp32 [B][q_len][H][D].  The workspace is sized
    by attn_decode_workspace_bytes(B * q_len, H, ...)."""
    B, Q, H = q.shape[0], q.shape[1], q.shape[2]
    ws = _dev(workspace, torch.uint8, "workspace") if workspace is not None else None
    nbytes = workspace.numel() if workspace is not None else 0
    _check(lib().attn_decode_multi_int8(pool.handle, layer, _dev(q, torch.float16, "q"), B, Q, H,
                                        _dev(seq_lens, torch.int32, "seq_lens"),
                                        _dev(page_table, torch.int32, "page_table"),
                                        page_table.shape[1], float(softmax_scale), n_splits,
                                        _dev(out, torch.float32, "out"), ws, nbytes,
                                        _stream(stream)), "attn_decode_multi_int8")


def attn_prefill_n_splits(pool, n_new, n_heads, start_pos):
    n = lib().attn_prefill_n_splits(pool.handle, n_new, n_heads, start_pos)
    if n < 0:
        raise Int8KVError(n, "attn_prefill_n_splits")
    return n


def attn_prefill_workspace_bytes(n_new, n_heads, n_kv_heads, head_dim, n_splits):
    out = _c_size(0)
    _check(lib().attn_prefill_workspace_bytes(n_new, n_heads, n_kv_heads, head_dim, n_splits,
                                              ctypes.byref(out)), "attn_prefill_workspace_bytes")
    return out.value


def attn_prefill_chunk_int8(pool, layer, q, start_pos, page_table, out, workspace=None,
                            softmax_scale=0.0, n_splits=0, stream=None):
    """q fp16 [n_new][H][D]; page_table int32 [max_pages] (one sequence); out fp32 [n_new][H][D]."""
    n_new, H = q.shape[0], q.shape[1]
    ws = _dev(workspace, torch.uint8, "workspace") if workspace is not None else None
    nbytes = workspace.numel() if workspace is not None else 0
    _check(lib().attn_prefill_chunk_int8(pool.handle, layer, _dev(q, torch.float16, "q"), n_new,
                                         H, start_pos, _dev(page_table, torch.int32, "page_table"),
                                         page_table.shape[-1], float(softmax_scale), n_splits,
                                         _dev(out, torch.float32, "out"), ws, nbytes,
                                         _stream(stream)), "attn_prefill_chunk_int8")


def kv_pool_set_decode_kernel(pool, kind):
    """kind: DECODE_AUTO, DECODE_WARP_MMA or DECODE_SIMT."""
    _check(lib().kv_pool_set_decode_kernel(pool.handle, int(kind)), "kv_pool_set_decode_kernel")


def _host_lens(seq_lens):
    lens = torch.as_tensor(seq_lens, dtype=torch.int32).cpu().contiguous()
    return lens, ctypes.c_void_p(lens.data_ptr())


def kv_pool_image_bytes(pool, seq_lens):
    """Bytes of the saved image of sequences of these lengths (a host sequence)."""
    lens, lp = _host_lens(seq_lens)
    out = _c_size(0)
    _check(lib().kv_pool_image_bytes(pool.handle, lens.numel(), lp, ctypes.byref(out)),
           "kv_pool_image_bytes")
    return out.value


def kv_pool_save(pool, seq_lens, page_table, staging=None, stream=None):
    """The saved image (bytes) of positions 0..L_b-1 of every layer of each sequence.
    seq_lens: host lengths; page_table: int32 [n_seqs][max_pages] on the device;
    staging: a device uint8 tensor of at least the image's bytes (allocated here
    when None)."""
    lens, lp = _host_lens(seq_lens)
    n = kv_pool_image_bytes(pool, lens)
    if staging is None:
        staging = torch.empty(max(n, 16), dtype=torch.uint8, device=page_table.device)
    host = torch.empty(max(n, 1), dtype=torch.uint8)
    _check(lib().kv_pool_save(pool.handle, lens.numel(), lp,
                              _dev(page_table, torch.int32, "page_table"), page_table.shape[1],
                              _dev(staging, torch.uint8, "staging"), staging.numel(),
                              ctypes.c_void_p(host.data_ptr()), host.numel(), _stream(stream)),
           "kv_pool_save")
    return bytes(host[:n].numpy())


def kv_pool_load(pool, image, page_table, staging=None, stream=None):
    """Load a saved image into the pool through page_table (int32 [n_seqs][max_pages]
    on the device); returns the sequences' lengths."""
    n_seqs = page_table.shape[0]
    buf = torch.frombuffer(bytearray(image), dtype=torch.uint8) if len(image) else \
        torch.zeros(1, dtype=torch.uint8)
    if staging is None:
        staging = torch.empty(max(len(image), 16), dtype=torch.uint8, device=page_table.device)
    lens = torch.zeros(max(n_seqs, 1), dtype=torch.int32)
    _check(lib().kv_pool_load(pool.handle, ctypes.c_void_p(buf.data_ptr()), len(image), n_seqs,
                              _dev(page_table, torch.int32, "page_table"), page_table.shape[1],
                              _dev(staging, torch.uint8, "staging"), staging.numel(),
                              ctypes.c_void_p(lens.data_ptr()), _stream(stream)), "kv_pool_load")
    return lens[:n_seqs].tolist()


def kv_pool_test_expire_waits(pool, max_polls):
    """Diagnostic: later decode calls arm their copy waits so that they expire after
    max_polls polls and report INT8KV_DEVERR_TIMEOUT (0 switches it off)."""
    _check(lib().kv_pool_test_expire_waits(pool.handle, int(max_polls)),
           "kv_pool_test_expire_waits")


def kv_pool_read_device_error(pool, stream=None):
    v = ctypes.c_int32(0)
    _check(lib().kv_pool_read_device_error(pool.handle, ctypes.byref(v), _stream(stream)),
           "kv_pool_read_device_error")
    return v.value


class KVPool:
    """Owns the device regions of a pool (torch allocations) and its descriptor."""

    def __init__(self, n_layers, n_kv_heads, head_dim, group_size, page_size, n_pages,
                 variant=K8V8, device=None):
        if isinstance(variant, str):
            variant = VARIANTS[variant]
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        shape = (n_layers, n_pages, n_kv_heads, page_size, head_dim)
        ng = head_dim // group_size
        sshape = (n_layers, n_pages, n_kv_heads, page_size, ng)
        k8 = variant in (K8V8, K8V16, K8V4)
        v8 = variant in (K8V8, K16V8)
        k4 = variant == Q4_0
        v4 = variant in (K8V4, Q4_0)
        self.k_store = torch.zeros(shape, dtype=torch.int8 if k8 else torch.float16, device=dev)
        self.v_store = torch.zeros(shape, dtype=torch.int8 if v8 else torch.float16, device=dev)
        self.k_scales = torch.zeros(sshape, dtype=torch.float16, device=dev) if k8 else None
        self.v_scales = torch.zeros(sshape, dtype=torch.float16, device=dev) if v8 else None
        if k4:   # 4-bit stores: two codes per byte, one fp16 scale per 32 values
            self.k_store = torch.zeros(shape[:-1] + (head_dim // 2,), dtype=torch.uint8, device=dev)
            self.k_scales = torch.zeros(shape[:-1] + (head_dim // 32,), dtype=torch.float16,
                                        device=dev)
        if v4:
            self.v_store = torch.zeros(shape[:-1] + (head_dim // 2,), dtype=torch.uint8, device=dev)
            self.v_scales = torch.zeros(shape[:-1] + (head_dim // 32,), dtype=torch.float16,
                                        device=dev)
        self.dev_error = torch.zeros(4, dtype=torch.int32, device=dev)
        for region, t in ((REGION_K_STORE, self.k_store), (REGION_V_STORE, self.v_store),
                          (REGION_K_SCALES, self.k_scales), (REGION_V_SCALES, self.v_scales)):
            want = int8kv_pool_region_bytes(n_layers, n_kv_heads, head_dim, group_size,
                                            page_size, n_pages, variant, region)
            have = 0 if t is None else t.numel() * t.element_size()
            assert want == have, (region, want, have)
        self.n_layers, self.n_kv_heads, self.head_dim = n_layers, n_kv_heads, head_dim
        self.group_size, self.page_size, self.n_pages, self.variant = (group_size, page_size,
                                                                       n_pages, variant)
        self.handle = kv_pool_create(n_layers, n_kv_heads, head_dim, group_size, page_size,
                                     n_pages, variant, self.k_store, self.v_store,
                                     self.k_scales, self.v_scales, self.dev_error)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.kv_pool_destroy(h)
            self.handle = None

    def set_decode_kernel(self, kind):
        kv_pool_set_decode_kernel(self, kind)

    def decode_workspace(self, batch, n_heads, n_splits):
        n = attn_decode_workspace_bytes(batch, n_heads, self.n_kv_heads, self.head_dim, n_splits)
        return torch.zeros(max(n, 16), dtype=torch.uint8, device=self.k_store.device)
