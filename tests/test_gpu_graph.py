"""CUDA-graph capture of the library's calls: a replayed step gives the same
bits as the eager call (the fused stack step, whose SWA launch is a
programmatic dependent of the Full split launch, and the split + merge
decode, whose merge launch is one)."""
import numpy as np
import pytest
import torch

import paged_hybrid_sliding_gb300 as phs
import synth
from gpu_util import dev

pytestmark = pytest.mark.gpu


def _layers(n_after, Hq, Hkv, D, layer_is_full, seed, W=128):
    B = len(n_after)
    bt, num_pages = synth.block_tables_from_permutation(synth.pages_needed(n_after), seed)
    rp = synth.ring_positions(B, W, seed + 1)
    layers = []
    for l, full in enumerate(layer_is_full):
        s = seed * 100 + 10 * l
        kw = dict(q=synth.normal_bf16((B, Hq, D), s, device="cuda"),
                  out=torch.zeros((B, Hq, D), dtype=torch.float32, device="cuda"),
                  k_new=synth.normal_bf16((B, Hkv, D), s + 1, device="cuda"),
                  v_new=synth.normal_bf16((B, Hkv, D), s + 2, device="cuda"))
        shape = (num_pages, Hkv, 16, D) if full else (B, Hkv, W, D)
        pool = (synth.normal_bf16(shape, s + 3, device="cuda"),
                synth.normal_bf16(shape, s + 4, device="cuda"))
        if full:
            kw["paged"] = phs.PagedPool(*pool)
        else:
            kw["ring"] = phs.RingPool(*pool)
        layers.append(phs.Layer(**kw))
    return layers, bt, rp


def test_fused_stack_graph_replay_equals_eager():
    n_after = np.array([40, 700, 3000, 5100], np.int32)   # multi-split Full requests
    Hq, Hkv, D = 8, 2, 64
    layers, bt, rp = _layers(n_after, Hq, Hkv, D, [1, 0, 1, 0, 0], seed=3)
    sl, btd, rpd = dev(n_after), dev(bt), dev(rp)
    ws = torch.empty(phs.hybrid_stack_fused_workspace_bytes(len(n_after), Hq, Hkv, D,
                                                            int(n_after.max()), 2),
                     dtype=torch.uint8, device="cuda")

    def step():
        phs.attn_decode_hybrid_stack_fused(layers, Hq, sl, int(n_after.max()), block_table=btd,
                                           ring_pos=rpd, workspace=ws)

    step()  # eager (the appends are idempotent: the same token into the same slot)
    torch.cuda.synchronize()
    eager = [L.out.clone() for L in layers]
    for L in layers:
        L.out.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for l, (L, e) in enumerate(zip(layers, eager)):
        assert torch.equal(L.out, e), l


def test_split_merge_decode_graph_replay_equals_eager():
    w = synth.paged_full(seed=12, B=12, lo=1000, hi=9000)
    Hq, Hkv, D = w.Hq, w.Hkv, w.D
    pool = phs.PagedPool(synth.normal_bf16((w.num_pages, Hkv, 16, D), 1, device="cuda"),
                         synth.normal_bf16((w.num_pages, Hkv, 16, D), 2, device="cuda"))
    q = synth.normal_bf16((w.B, Hq, D), 3, device="cuda")
    sl, bt = dev(w.n_after), dev(w.block_table)
    tps = 256  # several splits per request: the merge launch runs
    ws = torch.empty(phs.decode_workspace_bytes(w.B, Hq, Hkv, D, int(w.n_after.max()), tps),
                     dtype=torch.uint8, device="cuda")
    out = torch.zeros((w.B, Hq, D), dtype=torch.float32, device="cuda")

    def step():
        phs.attn_decode_full_paged(q, pool, bt, sl, int(w.n_after.max()), out=out,
                                   tokens_per_split=tps, workspace=ws)

    step()
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
