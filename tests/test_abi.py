"""The C ABI library loads and exports every entry point include/kvq.h declares (CPU only:
pure-host calls and argument checks that return before any CUDA call)."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")
LIB = os.path.join(ROOT, "flash_decode_quantized_gb300", "libkvq.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from flash_decode_quantized_gb300 import build
        build.build()
    return ctypes.CDLL(LIB)


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared()
    for n in ("kvq_store_create", "kvq_append", "kvq_flash_decode", "kvq_destroy"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (kvq_\w+)", out))
    missing = [n for n in declared() if n not in exported]
    assert not missing, missing
    for n in declared():
        getattr(lib, n)


def test_pure_host_calls(lib):
    from flash_decode_quantized_gb300 import kvq
    assert kvq.kvq_store_bytes("q8_0", 8, 128, 256, 10) == 10 * 8 * 256 * (128 + 8)
    assert kvq.kvq_store_bytes("q4s", 2, 256, 256, 1) == 2 * 256 * (128 + 16)
    assert kvq.kvq_store_bytes("bf16", 1, 64, 64, 3) == 3 * 64 * 128
    assert kvq.kvq_status_string(0) == "KVQ_OK"
    assert kvq.kvq_status_string(5) == "KVQ_ERR_WORKSPACE"
    for bad in [("q8_0", 8, 96, 256, 1), ("q8_0", 0, 128, 256, 1), ("q8_0", 8, 128, 100, 1),
                (7, 8, 128, 256, 1), ("q8_0", 8, 128, 256, 0)]:
        with pytest.raises(kvq.KvqError):
            kvq.kvq_store_bytes(*bad)


def test_null_arguments_rejected_before_any_cuda_call(lib):
    from flash_decode_quantized_gb300 import kvq
    L = kvq.lib
    assert L.kvq_append(None, None, 1, 1, None, None, 1, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_seq_lens_add(None, 1, 1, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_flash_decode(None, None, None, None, None, 1, kvq.CodecPair(2, 2), None, 1, 1,
                              0.0, 1, None, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_flash_decode_append(None, None, None, None, None, None, None, 1, kvq.CodecPair(2, 2),
                                     None, 1, 1, 0.0, 1, 1, None, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_dequantize(None, None, None, None, 1, 1, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_read_probe(None, 1024, None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_pointer_kind(None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_prefill_attention(None, None, None, None, None, 1, kvq.CodecPair(2, 2), None, 1, 1, 1,
                                   0.0, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_decode_workspace_bytes(None, None, 1, 1, 1, None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_store_get_error(None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_destroy(None) == kvq.KVQ_OK
    h = ctypes.c_void_p()
    d = kvq.StoreDesc(2, 8, 128, 256, 1)
    assert L.kvq_store_create(ctypes.byref(d), None, 0, ctypes.byref(h)) == kvq.KVQ_ERR_INVALID_ARG
    assert h.value is None
    assert isinstance(kvq.kvq_launch_count(), int)
    for bad in [(-1, -1), (0, -2)]:
        assert L.kvq_set_fault_injection(*bad) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_set_fault_injection(0, -1) == kvq.KVQ_OK   # the default: no injection
