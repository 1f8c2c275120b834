"""Programmatic dependent launch (PDL) and graph capture of a decode step on the GPU.

With PDL on, each kernel of the library may start launching while the previous one runs
and waits (griddepcontrol.wait) before reading its inputs, so the results must equal the
serialised launches bit for bit: an append followed at once by the decode that reads the
appended keys, repeated back to back, on both caches, eagerly and inside a CUDA graph.
Every step's output is also held to the oracle, which replays the same appends on a host
copy of the pool (a race that broke the serialised launches too would show there).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_gb300 as pkv
from paged_kv_gqa_gb300 import _build
from gpu_util import LSE_TOL, OUT_TOL, max_abs_diff
from workloads import bf16_bits, make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    lib = pkv.load()
    yield lib
    pkv.set_programmatic_launch(False)


class Step:
    """One decode iteration on the batch shape: write each sequence's newest key and value
    (the last slot of its length), then attend over all its keys."""

    def __init__(self, cache, seed, max_pages=None):
        spec = dict(B=8, Hq=32, Hkv=8, D=128, P=16, lens=("uniform", 200, 3000), seed=seed)
        if max_pages is not None:  # a table wider than the sequences (a pool sized for long contexts)
            spec["max_pages"] = max_pages
        c = make_case(spec, device="cuda")
        self.c = c
        self.cache = cache
        g = torch.Generator(device="cuda")
        g.manual_seed(seed + 1)
        self.steps = 6
        self.kn = [torch.randn(c.B, c.Hkv, c.D, generator=g, device="cuda").to(torch.bfloat16) for _ in range(self.steps)]
        self.vn = [torch.randn(c.B, c.Hkv, c.D, generator=g, device="cuda").to(torch.bfloat16) for _ in range(self.steps)]
        self.pos = (c.seq_lens - 1).to(torch.int32)
        if cache == "fp8":
            self.pools = list(pkv.quantize_pool_fp8(c.k_cache, c.v_cache))
        self.k0 = c.k_cache.clone()
        self.v0 = c.v_cache.clone()
        ws = pkv.paged_decode_attn_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.P, c.max_pages, cache=cache)
        self.ws = torch.zeros(ws, dtype=torch.uint8, device="cuda")
        self.out = torch.empty(self.steps, c.B, c.Hq, c.D, dtype=torch.bfloat16, device="cuda")
        self.lse = torch.empty(self.steps, c.B, c.Hq, dtype=torch.float32, device="cuda")

    def reset(self):
        # in place: a captured graph keeps the addresses of these tensors
        self.c.k_cache.copy_(self.k0)
        self.c.v_cache.copy_(self.v0)
        if self.cache == "fp8":
            for dst, src in zip(self.pools, pkv.quantize_pool_fp8(self.c.k_cache, self.c.v_cache)):
                dst.copy_(src)
        self.out.fill_(float("nan"))
        self.lse.fill_(float("nan"))

    def run(self, stream=None):
        c = self.c
        for i in range(self.steps):
            if self.cache == "fp8":
                pkv.paged_kv_append_fp8(self.kn[i], self.vn[i], c.block_table, self.pos, *self.pools, stream=stream)
                pkv.paged_decode_attn_fp8(c.q, *self.pools, c.block_table, c.seq_lens, c.scale, self.out[i],
                                          self.lse[i], self.ws, stream=stream)
            else:
                pkv.paged_kv_append(self.kn[i], self.vn[i], c.block_table, self.pos, c.k_cache, c.v_cache,
                                    stream=stream)
                pkv.paged_decode_attn(c.q, c.k_cache, c.v_cache, c.block_table, c.seq_lens, c.scale, self.out[i],
                                      self.lse[i], self.ws, stream=stream)


def assert_steps_match_oracle(st):
    """Replays the step's appends on the oracle's host copy of the pool (the fp8 pool made by
    the oracle's own quantiser) and holds each step's out and lse to the oracle bars."""
    c = st.c
    q, bt, sl = bf16_bits(c.q), c.block_table.cpu().numpy(), c.seq_lens.cpu().numpy()
    pos = st.pos.cpu().numpy()
    k, v = bf16_bits(st.k0), bf16_bits(st.v0)
    if st.cache == "fp8":
        (k8, ks), (v8, vs) = oracle.quantize_pool(k), oracle.quantize_pool(v)
    for i in range(st.steps):
        kn, vn = bf16_bits(st.kn[i]), bf16_bits(st.vn[i])
        if st.cache == "fp8":
            k8, v8, ks, vs, rej = oracle.kv_append_fp8(kn, vn, bt, pos, k8, v8, ks, vs)
            ro, rl = oracle.paged_decode_fp8(q, k8, v8, ks, vs, bt, sl, c.scale)
        else:
            k, v, rej = oracle.kv_append(kn, vn, bt, pos, k, v)
            ro, rl = oracle.paged_decode(q, k, v, bt, sl, c.scale)
        assert rej == 0
        eo = max_abs_diff(st.out[i].float().cpu().numpy(), ro)
        el = max_abs_diff(st.lse[i].cpu().numpy(), rl)
        assert eo <= OUT_TOL and el <= LSE_TOL, (i, eo, el)


@pytest.mark.parametrize("cache", ["bf16", "fp8"])
def test_pdl_results_equal_serialised_launches(cache):
    st = Step(cache, seed=11)
    pkv.set_programmatic_launch(False)
    st.reset()
    st.run()
    torch.cuda.synchronize()
    ref_o, ref_l = st.out.clone(), st.lse.clone()
    assert torch.isfinite(ref_o.float()).all()
    # each step's output depends on the key appended just before it
    assert not torch.equal(ref_o[0], ref_o[1])
    assert pkv.set_programmatic_launch(True) is False
    for _ in range(3):
        st.reset()
        st.run()
        torch.cuda.synchronize()
        assert torch.equal(st.out.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(st.lse.view(torch.int32), ref_l.view(torch.int32))
    assert pkv.pkv_check_status(st.ws) == 0
    pkv.set_programmatic_launch(False)
    assert_steps_match_oracle(st)


@pytest.mark.parametrize("cache", ["bf16", "fp8"])
def test_pdl_inside_a_cuda_graph(cache):
    st = Step(cache, seed=12)
    pkv.set_programmatic_launch(False)
    st.reset()
    st.run()
    torch.cuda.synchronize()
    ref_o, ref_l = st.out.clone(), st.lse.clone()
    pkv.set_programmatic_launch(True)
    st.reset()
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        st.run(stream=s)
    for _ in range(2):
        st.reset()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(st.out.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(st.lse.view(torch.int32), ref_l.view(torch.int32))
    pkv.set_programmatic_launch(False)
    assert pkv.pkv_check_status(st.ws) == 0
    assert_steps_match_oracle(st)


@pytest.mark.parametrize("cache", ["bf16", "fp8"])
def test_adaptive_splits_under_pdl_and_graph(cache):
    """The adaptive split count (each block reads every length before it sizes the splits) on a
    table far wider than the sequences, with PDL eagerly and inside a graph: equal bit for bit to
    the serialised launches of the same mode, and held to the oracle."""
    st = Step(cache, seed=13, max_pages=4096)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    c = st.c
    plan = pkv.plan_query(c.B, c.Hq, c.Hkv, c.D, c.P, c.max_pages, sms, cache=cache)
    assert plan["num_splits"] > 1 and plan["chunk_tokens"] > 2048, plan
    prev = pkv.set_adaptive_splits(True)
    try:
        pkv.set_programmatic_launch(False)
        st.reset()
        st.run()
        torch.cuda.synchronize()
        ref_o, ref_l = st.out.clone(), st.lse.clone()
        pkv.set_programmatic_launch(True)
        st.reset()
        st.run()
        torch.cuda.synchronize()
        assert torch.equal(st.out.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(st.lse.view(torch.int32), ref_l.view(torch.int32))
        st.reset()
        s = torch.cuda.Stream()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            st.run(stream=s)
        for _ in range(2):
            st.reset()
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(st.out.view(torch.int16), ref_o.view(torch.int16))
            assert torch.equal(st.lse.view(torch.int32), ref_l.view(torch.int32))
    finally:
        pkv.set_programmatic_launch(False)
        pkv.set_adaptive_splits(prev)
    assert pkv.pkv_check_status(st.ws) == 0
    assert_steps_match_oracle(st)
