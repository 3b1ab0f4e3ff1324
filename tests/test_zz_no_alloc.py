"""kvq_flash_decode_static_ws: the decode entry point for callers that cannot allocate.

Callers inside host callbacks, under a memory manager that owns all device memory, or
in loops that cannot afford cudaMalloc's synchronization get a decode call without a
workspace argument; it uses a fixed array in the library's device memory instead.  It runs
the same plan and the same kernels as kvq_flash_decode, so its output must match that
call bit for bit.  This file runs last (its name sorts last) and must pass both alone and
after the others.
"""

import numpy as np
import pytest
import torch

from kvq_testutil import assert_close, build_store, device_inputs, kvq, oracle_out
from workloads import make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", [2, 1])
@pytest.mark.parametrize("kc,vc", [("q8_0", "q8_0"), ("q4s", "q4s")])
def test_static_workspace_matches_allocating_entry_point(kc, vc, variant):
    inp = make_inputs([3000, 1200], 32, 8, 128, seed=31)
    k = kvq()
    ks = build_store(inp, kc, "k")
    vs = build_store(inp, vc, "v")
    q, sl, pt = device_inputs(inp)
    want = k.kvq_flash_decode(q, ks, vs, sl, pt, max_len_hint=3000, variant=variant)
    for _ in range(2):   # two calls in a row share and reuse the static array
        got = k.kvq_flash_decode_static_ws(q, ks, vs, sl, pt, max_len_hint=3000, variant=variant)
        assert k.kvq_store_get_error(ks) == 0 and k.kvq_store_get_error(vs) == 0
        assert torch.equal(got, want)   # same plan, same kernels: the same bits
    if variant == 2 and kc == "q8_0":
        assert_close(got.cpu().numpy(), oracle_out(inp, kc, vc), "static workspace vs oracle")


def test_rejected_call_enqueues_nothing():
    # a call that fails its host checks (here: a softmax scale that is not finite) returns
    # its error before touching the array; the next valid call is unaffected
    inp = make_inputs([2000], 16, 4, 128, seed=33)
    k = kvq()
    ks = build_store(inp, "q8_0", "k")
    vs = build_store(inp, "q8_0", "v")
    q, sl, pt = device_inputs(inp)
    first = k.kvq_flash_decode_static_ws(q, ks, vs, sl, pt, max_len_hint=2000)
    with pytest.raises(k.KvqError) as e:
        k.kvq_flash_decode_static_ws(q, ks, vs, sl, pt, max_len_hint=2000, softmax_scale=float("nan"))
    assert e.value.status == k.KVQ_ERR_INVALID_ARG
    again = k.kvq_flash_decode_static_ws(q, ks, vs, sl, pt, max_len_hint=2000)
    assert k.kvq_store_get_error(ks) == 0
    assert torch.equal(first, again)


def test_static_workspace_rejects_oversized_splits():
    inp = make_inputs([64], 8, 2, 128, seed=32)
    k = kvq()
    ks = build_store(inp, "q8_0", "k")
    vs = build_store(inp, "q8_0", "v")
    q, sl, pt = device_inputs(inp)
    big_q = torch.zeros((4096, 8, 128), dtype=torch.bfloat16, device="cuda")
    big_sl = torch.full((4096,), 64, dtype=torch.int32, device="cuda")
    big_pt = pt.expand(4096, -1).contiguous()
    with pytest.raises(k.KvqError) as e:
        k.kvq_flash_decode_static_ws(big_q, ks, vs, big_sl, big_pt, max_len_hint=256, chunk_tokens=64)
    assert e.value.status == k.KVQ_ERR_WORKSPACE
