"""Python binding of the kvq C ABI (include/kvq.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does nothing but
check Python-side types, pass device pointers / sizes / the current CUDA stream through
ctypes, and raise ``KvqError`` on a non-OK status.  All computation runs in the CUDA
kernels of libkvq.so; there is no fallback: importing this module without the built
library raises.  PyTorch is used only to allocate device memory and to name streams.
"""

from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvq.so")

KVQ_OK, KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_CUDA, KVQ_ERR_DEVICE_FAULT, \
    KVQ_ERR_WORKSPACE = range(6)
CODECS = {"bf16": 0, "f16": 1, "q8_0": 2, "q4s": 3}
DEVICE_FAULTS = {0: "ok", 1: "bad_page", 2: "bad_position", 3: "bad_seq_len", 4: "timeout",
                 5: "bad_workspace"}


class KvqError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call} -> {_status_string(status)}")


class StoreDesc(ctypes.Structure):
    _fields_ = [("codec", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int32)]


class CodecPair(ctypes.Structure):
    _fields_ = [("k", ctypes.c_int32), ("v", ctypes.c_int32)]


class DecodeOpts(ctypes.Structure):
    _fields_ = [("chunk_tokens", ctypes.c_int32), ("variant", ctypes.c_int32)]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libkvq.so is not built ({_LIB_PATH}); run "
                          "`python -m flash_decode_quantized_gb300.build`")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, Z, V = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
    sig = {
        "kvq_store_bytes": [ctypes.POINTER(StoreDesc), ctypes.POINTER(Z)],
        "kvq_store_create": [ctypes.POINTER(StoreDesc), P, Z, ctypes.POINTER(P)],
        "kvq_destroy": [P],
        "kvq_append": [P, P, I, I, P, P, I, V],
        "kvq_seq_lens_add": [P, I, I, V],
        "kvq_append_kv": [P, P, P, P, I, I, P, P, I, I, V],
        "kvq_decode_workspace_bytes": [P, P, I, I, I, ctypes.POINTER(DecodeOpts), ctypes.POINTER(Z)],
        "kvq_flash_decode": [P, P, P, P, P, I, CodecPair, P, I, I, ctypes.c_float, I,
                             ctypes.POINTER(DecodeOpts), P, Z, V],
        "kvq_store_get_error": [P, ctypes.POINTER(ctypes.c_int32)],
        "kvq_decode_workspace_init": [P, Z, V],
        "kvq_flash_decode_static_ws": [P, P, P, P, P, I, CodecPair, P, I, I, ctypes.c_float, I,
                                       ctypes.POINTER(DecodeOpts), V],
        "kvq_dequantize": [P, P, P, P, I, I, V],
        "kvq_read_probe": [P, Z, P, V],
        "kvq_pointer_kind": [P, ctypes.POINTER(ctypes.c_int32)],
        "kvq_prefill_attention": [P, P, P, P, P, I, CodecPair, P, I, I, I, ctypes.c_float, V],
        "kvq_flash_decode_multi": [P, P, P, P, P, I, CodecPair, P, I, I, I, ctypes.c_float, I,
                                   ctypes.POINTER(DecodeOpts), P, Z, V],
        "kvq_flash_decode_append": [P, P, P, P, P, P, P, I, CodecPair, P, I, I, ctypes.c_float, I, I,
                                    ctypes.POINTER(DecodeOpts), P, Z, V],
        "kvq_set_fault_injection": [ctypes.c_int32, ctypes.c_int32],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.kvq_launch_count.argtypes = []
    lib.kvq_launch_count.restype = ctypes.c_uint64
    lib.kvq_status_string.argtypes = [ctypes.c_int]
    lib.kvq_status_string.restype = ctypes.c_char_p
    return lib


lib = _load()


def _status_string(status: int) -> str:
    return lib.kvq_status_string(status).decode()


def _check(status: int, call: str) -> None:
    if status != KVQ_OK:
        raise KvqError(status, call)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def pointer_kind(ptr: int) -> int:
    """kvq_pointer_kind: 0 device memory, 1 host memory mapped at the same address, -1 other."""
    k = ctypes.c_int32(-1)
    _check(lib.kvq_pointer_kind(ctypes.c_void_p(ptr), ctypes.byref(k)), "kvq_pointer_kind")
    return k.value


def _ptr_io(t: torch.Tensor, dtype, name: str) -> int:
    """A step's input or output buffer: a CUDA tensor, or a pinned (page-locked) CPU tensor,
    which the kernel reads or writes in place through its device-visible mapping (the host
    transfer happens inside the step, with no copy-engine hand-off)."""
    if isinstance(t, torch.Tensor) and not t.is_cuda:
        if not t.is_pinned():
            raise TypeError(f"{name} must be a CUDA tensor or a pinned CPU tensor")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if pointer_kind(t.data_ptr()) != 1:
            raise TypeError(f"{name}: pinned memory not mapped into the device's address space")
        return t.data_ptr()
    return _ptr(t, dtype, name)


def _opts(chunk_tokens: int, variant: int):
    return ctypes.byref(DecodeOpts(int(chunk_tokens), int(variant)))


class Store:
    """A store handle plus the device buffer it wraps (owned by this object)."""

    def __init__(self, handle, buf, desc):
        self._h = handle
        self.buf = buf
        self.codec = {v: k for k, v in CODECS.items()}[desc.codec]
        self.num_kv_heads = desc.num_kv_heads
        self.head_dim = desc.head_dim
        self.page_size = desc.page_size
        self.num_pages = desc.num_pages

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("store was destroyed")
        return self._h

    def __del__(self):
        if getattr(self, "_h", None) is not None:
            lib.kvq_destroy(self._h)
            self._h = None


def _desc(codec, num_kv_heads, head_dim, page_size, num_pages) -> StoreDesc:
    return StoreDesc(CODECS[codec] if isinstance(codec, str) else int(codec), num_kv_heads,
                     head_dim, page_size, num_pages)


def kvq_store_bytes(codec, num_kv_heads: int, head_dim: int, page_size: int, num_pages: int) -> int:
    n = ctypes.c_size_t()
    _check(lib.kvq_store_bytes(ctypes.byref(_desc(codec, num_kv_heads, head_dim, page_size,
                                                  num_pages)), ctypes.byref(n)), "kvq_store_bytes")
    return n.value


def kvq_store_create(codec, num_kv_heads: int, head_dim: int, page_size: int, num_pages: int,
                     buf: torch.Tensor | None = None, device=None) -> Store:
    desc = _desc(codec, num_kv_heads, head_dim, page_size, num_pages)
    nbytes = kvq_store_bytes(codec, num_kv_heads, head_dim, page_size, num_pages)
    if buf is None:
        buf = torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")
    h = ctypes.c_void_p()
    _check(lib.kvq_store_create(ctypes.byref(desc), _ptr(buf, torch.uint8, "buf"), buf.numel(),
                                ctypes.byref(h)), "kvq_store_create")
    return Store(h, buf, desc)


def kvq_destroy(store: Store) -> None:
    if store._h is not None:
        _check(lib.kvq_destroy(store._h), "kvq_destroy")
        store._h = None


def kvq_append(store: Store, rows: torch.Tensor, seq_lens: torch.Tensor, page_table: torch.Tensor,
               stream=None) -> None:
    """rows: bf16 [B, n_new, Hkv, D]; writes row i of sequence b at seq_lens[b] + i."""
    if rows.dim() != 4 or rows.shape[2] != store.num_kv_heads or rows.shape[3] != store.head_dim:
        raise ValueError("rows must be [batch, n_new, num_kv_heads, head_dim]")
    bsz, n_new = rows.shape[0], rows.shape[1]
    if seq_lens.numel() != bsz or page_table.dim() != 2 or page_table.shape[0] != bsz:
        raise ValueError("seq_lens / page_table do not match the batch")
    _check(lib.kvq_append(store.handle, _ptr(rows, torch.bfloat16, "rows"), n_new, bsz,
                          _ptr(seq_lens, torch.int32, "seq_lens"),
                          _ptr(page_table, torch.int32, "page_table"), page_table.shape[1],
                          _stream(stream)), "kvq_append")


def kvq_append_kv(k_store: Store, v_store: Store, k_rows: torch.Tensor, v_rows: torch.Tensor,
                  seq_lens: torch.Tensor, page_table: torch.Tensor, advance: bool = True,
                  stream=None) -> None:
    """K and V rows (bf16 [B, n_new, Hkv, D] each) appended in one launch; with `advance`,
    seq_lens += n_new afterwards."""
    for name, rows, st in (("k_rows", k_rows, k_store), ("v_rows", v_rows, v_store)):
        if rows.dim() != 4 or rows.shape[2] != st.num_kv_heads or rows.shape[3] != st.head_dim:
            raise ValueError(f"{name} must be [batch, n_new, num_kv_heads, head_dim]")
    if k_rows.shape != v_rows.shape:
        raise ValueError("k_rows and v_rows differ in shape")
    bsz, n_new = k_rows.shape[0], k_rows.shape[1]
    if seq_lens.numel() != bsz or page_table.dim() != 2 or page_table.shape[0] != bsz:
        raise ValueError("seq_lens / page_table do not match the batch")
    _check(lib.kvq_append_kv(k_store.handle, v_store.handle, _ptr(k_rows, torch.bfloat16, "k_rows"),
                             _ptr(v_rows, torch.bfloat16, "v_rows"), n_new, bsz,
                             _ptr(seq_lens, torch.int32, "seq_lens"),
                             _ptr(page_table, torch.int32, "page_table"), page_table.shape[1],
                             1 if advance else 0, _stream(stream)), "kvq_append_kv")


def kvq_seq_lens_add(seq_lens: torch.Tensor, n: int, stream=None) -> None:
    _check(lib.kvq_seq_lens_add(_ptr(seq_lens, torch.int32, "seq_lens"), seq_lens.numel(), int(n),
                                _stream(stream)), "kvq_seq_lens_add")


def kvq_decode_workspace_bytes(k_store: Store, v_store: Store, batch: int, num_q_heads: int,
                               max_len_hint: int, chunk_tokens: int = 0, variant: int = 0) -> int:
    n = ctypes.c_size_t()
    _check(lib.kvq_decode_workspace_bytes(k_store.handle, v_store.handle, batch, num_q_heads,
                                          int(max_len_hint),
                                          _opts(chunk_tokens, variant), ctypes.byref(n)),
           "kvq_decode_workspace_bytes")
    return n.value


def kvq_flash_decode(q: torch.Tensor, k_store: Store, v_store: Store, seq_lens: torch.Tensor,
                     page_table: torch.Tensor, out: torch.Tensor | None = None,
                     softmax_scale: float = 0.0, max_len_hint: int | None = None,
                     workspace: torch.Tensor | None = None, chunk_tokens: int = 0,
                     variant: int = 0, stream=None) -> torch.Tensor:
    """q: bf16 [B, Hq, D] -> out fp32 [B, Hq, D].  max_len_hint defaults to the page
    table's capacity (max_pages * page_size)."""
    bsz, hq, dim = q.shape
    max_pages = page_table.shape[1]
    if max_len_hint is None:
        max_len_hint = max_pages * k_store.page_size
    if out is None:
        out = torch.empty((bsz, hq, dim), dtype=torch.float32, device=q.device)
    if workspace is None:   # (a given workspace is checked by the library itself)
        need = kvq_decode_workspace_bytes(k_store, v_store, bsz, hq, max_len_hint, chunk_tokens, variant)
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    codec = CodecPair(CODECS[k_store.codec], CODECS[v_store.codec])
    _check(lib.kvq_flash_decode(_ptr(q, torch.bfloat16, "q"), k_store.handle, v_store.handle,
                                _ptr(seq_lens, torch.int32, "seq_lens"),
                                _ptr(page_table, torch.int32, "page_table"), max_pages, codec,
                                _ptr(out, torch.float32, "out"), bsz, hq, float(softmax_scale),
                                int(max_len_hint), _opts(chunk_tokens, variant),
                                _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                                _stream(stream)), "kvq_flash_decode")
    return out


def kvq_flash_decode_multi(q: torch.Tensor, k_store: Store, v_store: Store, seq_lens: torch.Tensor,
                           page_table: torch.Tensor, out: torch.Tensor | None = None,
                           softmax_scale: float = 0.0, max_len_hint: int | None = None,
                           workspace: torch.Tensor | None = None, chunk_tokens: int = 0,
                           variant: int = 0, stream=None) -> torch.Tensor:
    """q: bf16 [B, Hq, T, D] (T query tokens per sequence, the last T positions being the
    drafts) -> out fp32 [B, Hq, T, D]; token i attends to positions < seq_len - T + 1 + i."""
    bsz, hq, t, dim = q.shape
    max_pages = page_table.shape[1]
    if max_len_hint is None:
        max_len_hint = max_pages * k_store.page_size
    if out is None:
        out = torch.empty((bsz, hq, t, dim), dtype=torch.float32, device=q.device)
    need = kvq_decode_workspace_bytes(k_store, v_store, bsz, hq * t, max_len_hint, chunk_tokens, variant)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    codec = CodecPair(CODECS[k_store.codec], CODECS[v_store.codec])
    _check(lib.kvq_flash_decode_multi(_ptr(q, torch.bfloat16, "q"), k_store.handle, v_store.handle,
                                      _ptr(seq_lens, torch.int32, "seq_lens"),
                                      _ptr(page_table, torch.int32, "page_table"), max_pages, codec,
                                      _ptr(out, torch.float32, "out"), bsz, hq, t, float(softmax_scale),
                                      int(max_len_hint), _opts(chunk_tokens, variant),
                                      _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                                      _stream(stream)), "kvq_flash_decode_multi")
    return out


class DecodeAppendStep:
    """kvq_flash_decode_append bound once to fixed buffers (the serving pattern: each step
    refills q / k_new / v_new in place and calls the step).  Arguments are checked and
    marshalled here once; a call is one library call.  q, k_new, v_new and out may be pinned
    CPU tensors: the step then reads its inputs from, and writes its output to, host memory
    itself (zero-copy), so a serving loop needs no separate copies around the call."""

    def __init__(self, q, k_new, v_new, k_store, v_store, seq_lens, page_table, out, workspace,
                 max_len_hint, advance=True, softmax_scale=0.0, chunk_tokens=0, variant=0, stream=None):
        bsz, hq, dim = q.shape
        for name, t, st in (("k_new", k_new, k_store), ("v_new", v_new, v_store)):
            if t.dim() != 3 or t.shape[0] != bsz or t.shape[1] != st.num_kv_heads or t.shape[2] != st.head_dim:
                raise ValueError(f"{name} must be [B, Hkv, D] = [{bsz}, {st.num_kv_heads}, {st.head_dim}]")
        if out.shape != (bsz, hq, dim):
            raise ValueError("out must be [B, Hq, D]")
        self._keep = (q, k_new, v_new, k_store, v_store, seq_lens, page_table, out, workspace)
        self._opts = _opts(chunk_tokens, variant)
        self._args = (_ptr_io(q, torch.bfloat16, "q"), _ptr_io(k_new, torch.bfloat16, "k_new"),
                      _ptr_io(v_new, torch.bfloat16, "v_new"), k_store.handle, v_store.handle,
                      _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(page_table, torch.int32, "page_table"),
                      page_table.shape[1], CodecPair(CODECS[k_store.codec], CODECS[v_store.codec]),
                      _ptr_io(out, torch.float32, "out"), bsz, hq, float(softmax_scale), int(max_len_hint),
                      1 if advance else 0, self._opts, _ptr(workspace, torch.uint8, "workspace"),
                      workspace.numel())
        self._stream = None if stream is None else _stream(stream)   # None: current at each call
        self.out = out

    def __call__(self):
        st = self._stream if self._stream is not None else torch.cuda.current_stream().cuda_stream
        status = lib.kvq_flash_decode_append(*self._args, st)
        if status != KVQ_OK:
            raise KvqError(status, "kvq_flash_decode_append")
        return self.out


def kvq_prefill_attention(q: torch.Tensor, k_store: Store, v_store: Store, seq_lens: torch.Tensor,
                          page_table: torch.Tensor, out: torch.Tensor | None = None,
                          softmax_scale: float = 0.0, stream=None) -> torch.Tensor:
    """q: bf16 [B, T, Hq, D], the last T positions of each sequence (already appended) ->
    out fp32 [B, T, Hq, D]; token i attends to positions <= seq_len - T + i."""
    bsz, t, hq, dim = q.shape
    if out is None:
        out = torch.empty((bsz, t, hq, dim), dtype=torch.float32, device=q.device)
    codec = CodecPair(CODECS[k_store.codec], CODECS[v_store.codec])
    _check(lib.kvq_prefill_attention(_ptr(q, torch.bfloat16, "q"), k_store.handle, v_store.handle,
                                     _ptr(seq_lens, torch.int32, "seq_lens"),
                                     _ptr(page_table, torch.int32, "page_table"), page_table.shape[1], codec,
                                     _ptr(out, torch.float32, "out"), bsz, hq, t, float(softmax_scale),
                                     _stream(stream)), "kvq_prefill_attention")
    return out


def kvq_flash_decode_append(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                            k_store: Store, v_store: Store, seq_lens: torch.Tensor,
                            page_table: torch.Tensor, advance: bool = True,
                            out: torch.Tensor | None = None, softmax_scale: float = 0.0,
                            max_len_hint: int | None = None, workspace: torch.Tensor | None = None,
                            chunk_tokens: int = 0, variant: int = 0, stream=None) -> torch.Tensor:
    """One decode step with the append fused in: k_new, v_new (bf16 [B, Hkv, D]) are
    written at position seq_lens[b], q attends over seq_lens[b] + 1 tokens, and with
    `advance` seq_lens[b] += 1 on the device."""
    bsz, hq, dim = q.shape
    for name, t, st in (("k_new", k_new, k_store), ("v_new", v_new, v_store)):
        if t.dim() != 3 or t.shape[0] != bsz or t.shape[1] != st.num_kv_heads or t.shape[2] != st.head_dim:
            raise ValueError(f"{name} must be [B, Hkv, D] = [{bsz}, {st.num_kv_heads}, {st.head_dim}]")
    max_pages = page_table.shape[1]
    if max_len_hint is None:
        max_len_hint = max_pages * k_store.page_size
    if out is None:
        out = torch.empty((bsz, hq, dim), dtype=torch.float32, device=q.device)
    if workspace is None:   # (a given workspace is checked by the library itself)
        need = kvq_decode_workspace_bytes(k_store, v_store, bsz, hq, max_len_hint, chunk_tokens, variant)
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    codec = CodecPair(CODECS[k_store.codec], CODECS[v_store.codec])
    _check(lib.kvq_flash_decode_append(_ptr(q, torch.bfloat16, "q"), _ptr(k_new, torch.bfloat16, "k_new"),
                                       _ptr(v_new, torch.bfloat16, "v_new"), k_store.handle, v_store.handle,
                                       _ptr(seq_lens, torch.int32, "seq_lens"),
                                       _ptr(page_table, torch.int32, "page_table"), max_pages, codec,
                                       _ptr(out, torch.float32, "out"), bsz, hq, float(softmax_scale),
                                       int(max_len_hint), 1 if advance else 0, _opts(chunk_tokens, variant),
                                       _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                                       _stream(stream)), "kvq_flash_decode_append")
    return out


def kvq_flash_decode_static_ws(q: torch.Tensor, k_store: Store, v_store: Store,
                               seq_lens: torch.Tensor, page_table: torch.Tensor,
                               out: torch.Tensor | None = None, softmax_scale: float = 0.0,
                               max_len_hint: int | None = None, chunk_tokens: int = 0,
                               variant: int = 0, stream=None) -> torch.Tensor:
    """kvq_flash_decode whose workspace is the library's fixed device array (no
    allocation by the library; `out` is allocated here only when not given)."""
    bsz, hq, dim = q.shape
    max_pages = page_table.shape[1]
    if max_len_hint is None:
        max_len_hint = max_pages * k_store.page_size
    if out is None:
        out = torch.empty((bsz, hq, dim), dtype=torch.float32, device=q.device)
    codec = CodecPair(CODECS[k_store.codec], CODECS[v_store.codec])
    _check(lib.kvq_flash_decode_static_ws(_ptr(q, torch.bfloat16, "q"), k_store.handle, v_store.handle,
                                          _ptr(seq_lens, torch.int32, "seq_lens"),
                                          _ptr(page_table, torch.int32, "page_table"), max_pages, codec,
                                          _ptr(out, torch.float32, "out"), bsz, hq, float(softmax_scale),
                                          int(max_len_hint), _opts(chunk_tokens, variant), _stream(stream)),
           "kvq_flash_decode_static_ws")
    return out


def kvq_dequantize(src: Store, dst: Store, seq_lens: torch.Tensor, page_table: torch.Tensor,
                   stream=None) -> None:
    """Separate dequantize pass: rows [0, seq_lens[b]) of the quantized store `src` rewritten
    into the 16-bit store `dst` (the unfused comparison arm)."""
    _check(lib.kvq_dequantize(src.handle, dst.handle, _ptr(seq_lens, torch.int32, "seq_lens"),
                              _ptr(page_table, torch.int32, "page_table"), page_table.shape[1],
                              seq_lens.shape[0], _stream(stream)), "kvq_dequantize")


def kvq_read_probe(buf: torch.Tensor, sink: torch.Tensor, stream=None) -> None:
    """Reads every byte of the (contiguous, 16-byte aligned) device tensor `buf` once."""
    _check(lib.kvq_read_probe(ctypes.c_void_p(buf.data_ptr()), buf.numel() * buf.element_size(),
                              _ptr(sink, torch.int32, "sink"), _stream(stream)), "kvq_read_probe")


def kvq_decode_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    """Zeroes a decode workspace (required once before its first use)."""
    _check(lib.kvq_decode_workspace_init(_ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                                         _stream(stream)), "kvq_decode_workspace_init")


def kvq_store_get_error(store: Store) -> int:
    """Synchronizes; returns (and clears) the first device fault code recorded, or 0."""
    code = ctypes.c_int32()
    st = lib.kvq_store_get_error(store.handle, ctypes.byref(code))
    if st not in (KVQ_OK, KVQ_ERR_DEVICE_FAULT):
        raise KvqError(st, "kvq_store_get_error")
    return code.value


def kvq_launch_count() -> int:
    return int(lib.kvq_launch_count())


def kvq_set_fault_injection(wait_limit: int, skip_tile: int) -> None:
    """Test hook for the device-timeout path; (0, -1) restores normal operation."""
    _check(lib.kvq_set_fault_injection(int(wait_limit), int(skip_tile)), "kvq_set_fault_injection")


def kvq_status_string(status: int) -> str:
    return _status_string(status)
