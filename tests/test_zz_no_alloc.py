"""kv_attend_decode_noalloc: decode attention for callers that cannot allocate device memory around a call. One
example is a serving engine whose memory planner owns the whole GPU and hands a kernel library only pointers
and a stream. Another is code that runs inside an allocator or memory-pool callback, where calling cudaMalloc
again would re-enter the allocator. The entry point keeps its scratch in one static device array of the library.
Its split plan and its kernels are those of kv_attend_decode, so its results must equal those of
kv_attend_decode with a caller workspace bit for bit, call after call, whatever a previous call left in that
array; both must also match the oracle.

This file is collected last so that a failure here stops a `-x` run only after every other test ran."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from transform_coded_kv_02_b300 import kvtc, synth

import gpu_helpers as G

pytestmark = pytest.mark.gpu
DEC_TOL = 2e-3


def _case(name, T, B, bits, seq_lens):
    w = synth.WORKLOADS[name]
    L = synth.make_layer(w, T=T, B=B, steps=1)
    sets = G.calibrate_oracle(L, bits, bits)
    P = G.lib_params(sets)
    rk, rv = G.oracle_cache(synth.as_float(L.k), synth.as_float(L.v), sets, L.per_seq_params, T)
    return w, L, P, rk, rv, seq_lens, sets


def _both(case):
    """Output of the workspace entry point and of the no-allocation entry point on the same inputs, and the
    oracle's decode of the same records."""
    w, L, P, rk, rv, seq_lens, sets = case
    B, Hkv, T_cap, _ = rk.shape
    tk, tv = G.dev_u32(rk), G.dev_u32(rv)
    cache = kvtc.make_cache(tk, tv, B, Hkv, T_cap, L.per_seq_params)
    q = G.to_dev_storage(L.q[0])
    sl = torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(w.d)
    ref = torch.full((B, w.Hq, w.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.zeros(kvtc.kv_decode_workspace_bytes(P, B, Hkv, w.Hq, T_cap), dtype=torch.uint8, device="cuda")
    kvtc.kv_attend_decode(P, cache, q, B, w.Hq, sl, scale, ref, ws)
    got = torch.full_like(ref, float("nan"))
    kvtc.kv_attend_decode_noalloc(P, cache, q, B, w.Hq, sl, scale, got)
    assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
    ora = G.oracle_decode(rk, rv, L.q[0], seq_lens, sets, w.Hq, L.per_seq_params)
    return got.cpu().numpy(), ref.cpu().numpy(), ora


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    # two different shapes back to back: the second call runs over whatever the first left in the scratch
    cases = [_case("llama_long_128k", 2048, 1, 1.33, [2000]),
             _case("qwen_batched_8k", 512, 2, 3.0, [512, 301])]
    for case in cases + cases[:1]:
        got, ref, ora = _both(case)
        assert np.all(np.isfinite(got))
        assert np.array_equal(got, ref), np.abs(got - ref).max()
        err = G.rel_l2_rows(got.astype(np.float64), ora)
        assert err.max() <= DEC_TOL, err


def test_noalloc_rejects_shapes_beyond_its_scratch():
    w, L, P, rk, rv, _, _ = _case("llama_long_128k", 64, 1, 1.33, [64])
    B, Hkv, T_cap = 256, w.Hkv, 64
    assert kvtc.kv_decode_workspace_bytes(P, B, Hkv, w.Hq, T_cap) > kvtc.NOALLOC_SCRATCH_BYTES
    tk = torch.zeros((B, Hkv, T_cap, P.record_words(0)), dtype=torch.int32, device="cuda")
    tv = torch.zeros(G.value_cache_shape(B, Hkv, T_cap, P.record_words(1)), dtype=torch.int32, device="cuda")
    cache = kvtc.make_cache(tk, tv, B, Hkv, T_cap)
    q = torch.zeros((B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    sl = torch.full((B,), T_cap, dtype=torch.int32, device="cuda")
    out = torch.zeros((B, w.Hq, w.d), dtype=torch.float32, device="cuda")
    with pytest.raises(kvtc.KvError) as e:
        kvtc.kv_attend_decode_noalloc(P, cache, q, B, w.Hq, sl, 1.0 / math.sqrt(w.d), out)
    assert e.value.status == kvtc.KV_ERR_INVALID_ARG
    assert "scratch" in str(e.value)
    assert kvtc.kv_check_status() == kvtc.KV_OK
