"""Streams and graphs: CUDA-graph capture of the entry points, as a serving loop
records prefill, backward and decode once and replays them, and calls on two
unordered streams at once.  Every call's workspace is stream-ordered (allocated and
freed on the call's stream) and the backward's kernels are chained by programmatic
launches, so a capture records memory nodes and programmatic edges; replays and
concurrent calls must reproduce the eager, sequential calls' bits."""

import pytest
import torch

from exact_attention_43_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bits(x):
    return x.view(torch.int16) if x.element_size() == 2 else x.view(torch.int32)


def test_graph_replay_matches_eager():
    import exact_attention_43_gb300 as ea

    dev = torch.device("cuda", 0)
    B, Hq, Hkv, S, D = 2, 4, 2, 384, 128  # GQA 2, a ragged last tile
    q, k, v = wl.fwd_inputs(B, Hq, Hkv, S, S, D, seed=wl.SEED_BASE + 300, device=dev)
    dout = wl.normal(tuple(q.shape), seed=wl.SEED_BASE + 301, device=dev)
    dq_in, k_cache, v_cache, lens = wl.decode_inputs(3, 8, 2, 1024, D, [1000, 17, 512],
                                                     seed=wl.SEED_BASE + 302, device=dev)
    lens = lens.to(dev)
    scale = D ** -0.5

    def alloc():
        return (torch.empty_like(q), torch.empty((B, Hq, S), dtype=torch.float32, device=dev),
                torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(dq_in))

    def run(outs):
        o, lse, dq, dk, dv, od = outs
        ea.attn_fwd(q, k, v, causal=True, scale=scale, out=o, lse=lse)
        ea.attn_bwd(q, k, v, o, lse, dout, causal=True, scale=scale, dq=dq, dk=dk, dv=dv)
        ea.attn_decode(dq_in, k_cache, v_cache, lens, num_splits=4, out=od)

    eager = alloc()
    run(eager)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0

    graphed = alloc()
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run(graphed)
    torch.cuda.synchronize()
    for _ in range(3):
        for t in graphed:
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert ea.check_device_status() == 0
        for name, a, b in zip(("o", "lse", "dq", "dk", "dv", "decode o"), eager, graphed):
            assert torch.equal(_bits(a), _bits(b)), name


def test_concurrent_streams_match_sequential():
    """Prefill and backward calls on two unordered streams at once: every call keeps its
    work counters and row terms in its own stream-ordered workspace, so the results
    are those of the same calls made one after another."""
    import exact_attention_43_gb300 as ea

    dev = torch.device("cuda", 0)
    cases = [(1, 8, 8, 1024), (2, 8, 2, 640)]  # B, Hq, Hkv, S
    inputs = []
    for n, (B, Hq, Hkv, S) in enumerate(cases):
        q, k, v = wl.fwd_inputs(B, Hq, Hkv, S, S, 128, seed=wl.SEED_BASE + 310 + 3 * n, device=dev)
        dout = wl.normal(tuple(q.shape), seed=wl.SEED_BASE + 311 + 3 * n, device=dev)
        inputs.append((q, k, v, dout))

    def run(q, k, v, dout):
        o, lse = ea.attn_fwd(q, k, v, causal=True)
        dq, dk, dv = ea.attn_bwd(q, k, v, o, lse, dout, causal=True)
        return o, lse, dq, dk, dv

    ref = [run(*x) for x in inputs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(device=dev) for _ in inputs]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    got = []
    for _ in range(3):
        outs = []
        for s, x in zip(streams, inputs):
            with torch.cuda.stream(s):
                outs.append(run(*x))
        torch.cuda.synchronize()
        got.append(outs)
    assert ea.check_device_status() == 0
    for outs in got:
        for r, g in zip(ref, outs):
            for a, b in zip(r, g):
                assert torch.equal(_bits(a), _bits(b))
