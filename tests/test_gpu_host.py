"""GPU tests of sa_attn_fwd_host: the path on pinned host tensors.

Each chunk of (batch, kv head) pairs is computed by the same kernels as the
device-buffer calls, and every head's result depends only on that head's
inputs (and its kv head's smooth-K mean), so the host path must reproduce
the device path bit for bit -- however the problem is chunked -- except
where the library's chunking of the NVFP4 path runs a small last chunk with
split-KV: the P quantisation is per key tile, so that changes only the
float32 summation order, and the float32 results agree to far below the
bf16 spacing.  The device path
itself is checked against the oracle in test_gpu_attn.py.  Argument errors
(pageable memory, a short workspace) are reported before anything is
enqueued.
"""

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    import quantized_attention_x16_gb300 as m
    return m


def device_path(sa, x, causal, mode, out_dtype):
    q, k, v = (x[n].cuda() for n in "qkv")
    if mode == "bf16":
        o = sa.sa_attn_fwd(q, k, v, causal=causal, mode="bf16", out_dtype=out_dtype)
    else:
        o = sa.sa_attn_fwd(sa.sa_quantize(q, k, v), causal=causal, mode="nvfp4", out_dtype=out_dtype)
    torch.cuda.synchronize()
    return o.cpu()


def host_path(sa, x, causal, mode, out_dtype, chunk_pairs):
    hq, hk, hv = (x[n].pin_memory() for n in "qkv")
    o = sa.sa_attn_fwd_host(hq, hk, hv, causal=causal, mode=mode, out_dtype=out_dtype, chunk_pairs=chunk_pairs)
    torch.cuda.current_stream().synchronize()
    assert sa.sa_last_device_error() == sa.SA_OK
    return o


CASES = [
    dict(W.spec("causal_gqa"), B=2, H=6, Hkv=3, L=384, seed=21),          # 6 pairs, G = 2, causal
    dict(W.spec("llm_prefill"), B=3, H=1, Hkv=1, L=512, seed=22),         # 3 pairs: ragged last chunk
    dict(W.spec("dit_video"), B=1, H=4, Hkv=2, L=256, d=64, seed=23),     # d = 64
    dict(W.spec("llm_prefill"), B=2, H=2, Hkv=2, L=300, seed=24),         # ragged L
    dict(W.spec("llm_prefill"), B=1, H=4, Hkv=4, L=2048, seed=25),        # library chunks split-KV
    dict(W.spec("causal_gqa"), B=1, H=8, Hkv=4, L=2100, seed=26),         # split-KV, causal, ragged
]


def _id(w):
    return f"B{w['B']}H{w['H']}K{w['Hkv']}L{w['L']}d{w['d']}{'c' if w['causal'] else ''}"


@pytest.mark.parametrize("chunk_pairs", [1, 2])
@pytest.mark.parametrize("mode", ["nvfp4", "bf16"])
@pytest.mark.parametrize("w", CASES, ids=_id)
def test_host_path_matches_device_path_bitwise(sa, w, mode, chunk_pairs):
    x = W.make_inputs(w)
    ref = device_path(sa, x, w["causal"], mode, torch.bfloat16)
    got = host_path(sa, x, w["causal"], mode, torch.bfloat16, chunk_pairs)
    assert got.dtype == torch.bfloat16 and tuple(got.shape) == tuple(ref.shape)
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("w", CASES, ids=_id)
def test_host_path_library_chunking_bf16_bitwise(sa, w):
    x = W.make_inputs(w)
    ref = device_path(sa, x, w["causal"], "bf16", torch.bfloat16)
    got = host_path(sa, x, w["causal"], "bf16", torch.bfloat16, 0)
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("w", CASES, ids=_id)
def test_host_path_library_chunking_nvfp4(sa, w):
    """chunk_pairs 0, NVFP4: split-KV chunks differ from the device path only
    in float32 summation order (P is quantised per key tile, whatever the
    running maximum), so the float32 outputs agree to a few float32 ulps of
    max|O|; unsplit chunks are bit-identical."""
    x = W.make_inputs(w)
    ref = device_path(sa, x, w["causal"], "nvfp4", torch.float32)
    got = host_path(sa, x, w["causal"], "nvfp4", torch.float32, 0)
    assert got.dtype == torch.float32 and tuple(got.shape) == tuple(ref.shape)
    err = (got - ref).abs().max().item()
    assert err <= 1e-5 * ref.abs().max().item(), err
    assert torch.isfinite(got).all()


def test_host_path_fp32_output_and_repeated_calls(sa):
    w = CASES[0]
    x = W.make_inputs(w)
    ref = device_path(sa, x, w["causal"], "nvfp4", torch.float32)
    hq, hk, hv = (x[n].pin_memory() for n in "qkv")
    need = sa.sa_attn_fwd_host_workspace_bytes(w["B"], w["H"], w["Hkv"], w["L"], w["d"], "nvfp4",
                                               torch.float32, 1)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    outs = [sa.sa_attn_fwd_host(hq, hk, hv, causal=True, mode="nvfp4", out_dtype=torch.float32, workspace=ws,
                                chunk_pairs=1) for _ in range(3)]   # back to back on one workspace
    torch.cuda.current_stream().synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int32), ref.view(torch.int32))


def test_host_path_rejects_bad_arguments(sa):
    w = CASES[1]
    x = W.make_inputs(w)
    hq, hk, hv = (x[n].pin_memory() for n in "qkv")
    B, H, L, d = hq.shape
    lib = sa.lib
    import ctypes
    o = torch.empty_like(hq).pin_memory()
    need = sa.sa_attn_fwd_host_workspace_bytes(B, H, 1, L, d, "nvfp4")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())      # noqa: E731
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    pageable = x["q"].contiguous()                    # not page-locked
    assert lib.sa_attn_fwd_host(p(pageable), p(hk), p(hv), p(o), B, H, 1, L, d, 0, 1, p(ws), need, 0, s) == \
        sa.SA_ERR_INVALID_ARG
    assert lib.sa_attn_fwd_host(p(hq), p(hk), p(hv), p(o), B, H, 1, L, d, 0, 1, p(ws), need - 256, 0, s) == \
        sa.SA_ERR_INVALID_ARG
    assert lib.sa_attn_fwd_host(p(hq), p(hk), p(hv), p(o), B, H, 1, L, 96, 0, 1, p(ws), need, 0, s) == \
        sa.SA_ERR_UNSUPPORTED                          # head dimension 96
    assert lib.sa_attn_fwd_host(p(hq), p(hk), p(hv), p(o), B, H, 1, L + 64, d, 0, 1, p(ws), need, 0, s) == \
        sa.SA_ERR_INVALID_ARG                          # a longer (ragged) problem needs a larger workspace
    assert lib.sa_attn_fwd_host(p(hq), p(hk), p(hv), p(o), B, H, 1, L, d, 0, 7, p(ws), need, 0, s) == \
        sa.SA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == sa.SA_OK


@pytest.mark.parametrize("mode", ["nvfp4", "bf16"])
def test_host_path_overlapped_back_to_back_calls(sa, mode):
    """SA_HOST_OVERLAP: calls queued back to back on one workspace, each on
    other inputs, each copy-in free to start before the previous call ends;
    every output must equal its own device-path result."""
    ws_case = dict(W.spec("llm_prefill"), B=2, H=4, Hkv=2, L=1000)
    xs = [W.make_inputs(dict(ws_case, seed=40 + i)) for i in range(4)]
    refs = [device_path(sa, x, False, mode, torch.bfloat16) for x in xs]
    need = sa.sa_attn_fwd_host_workspace_bytes(2, 4, 2, 1000, 128, mode)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    hs = [{n: x[n].pin_memory() for n in "qkv"} for x in xs]
    outs = []
    for _ in range(2):
        for h in hs:
            outs.append(sa.sa_attn_fwd_host(h["q"], h["k"], h["v"], mode=mode, workspace=ws, overlap=True))
    torch.cuda.current_stream().synchronize()
    assert sa.sa_last_device_error() == sa.SA_OK
    for i, o in enumerate(outs):
        ref = refs[i % len(refs)]
        if mode == "bf16":
            assert torch.equal(o.view(torch.int16), ref.view(torch.int16)), i
        else:   # split-KV chunks of the library's chunking: float32 summation order only
            assert (o.float() - ref.float()).abs().max().item() <= 2 ** -7 * ref.float().abs().max().item(), i
