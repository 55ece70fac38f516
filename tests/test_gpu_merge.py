"""The persistent decode kernel writes a partial (m, l, acc) for every
sequence split across CTAs and its merge kernel combines them.  These cases
stress that hand-off: a sequence spread over every CTA (more partials than
one round trip of the merge takes), more CTAs than blocks (CTAs with empty
ranges inside a sequence's span), a workspace full of garbage, and
CUDA-graph replays of one captured call."""
import numpy as np
import pytest
import torch

import workloads as W
from tests import pipeline as PL
from tests.test_gpu_decode import _check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_num_gb300 as P
    P.lib()
    return P


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
def test_one_sequence_over_every_cta(pkv, orc, kind):
    if kind == "bf16":
        w = W.gqa_bf16(batch=1, ctx_lo=30000, ctx_hi=30000, seed=260)
    else:
        w = W.fp8_long(batch=1, ctx_lo=20000, ctx_hi=20000, calib_tokens=64, seed=261)
    cache, out = PL.gpu_run(w, pkv)
    assert pkv.decode_launches(w.q.cuda(), cache, w.block_tables.cuda()) == 2
    _check(w, out, PL.oracle_decode(w, orc, PL.oracle_caches(w, orc)))


def test_more_ctas_than_blocks(pkv, orc):
    """Three blocks, a grid of eight CTAs (table capacity 8 blocks): CTAs 3,
    4 and 6 get empty ranges inside the sequence's span."""
    w = W.gqa_bf16(batch=1, ctx_lo=40, ctx_hi=40, seed=262)
    bt = torch.zeros((1, 8), dtype=torch.int32)
    bt[0, :w.block_tables.shape[1]] = w.block_tables[0]
    w.block_tables = bt
    _, out = PL.gpu_run(w, pkv)
    _check(w, out, PL.oracle_decode(w, orc, PL.oracle_caches(w, orc)))


def test_garbage_workspace_and_reuse(pkv):
    """Any workspace contents, and the same workspace over several calls,
    give the same bits as a fresh zeroed one."""
    w = W.gqa_bf16(batch=6, ctx_lo=100, ctx_hi=3000, seed=263)
    cache, ref = PL.gpu_run(w, pkv)
    q, bt, cl = w.q.cuda(), w.block_tables.cuda(), w.context_lens.cuda()
    n = pkv.decode_workspace_bytes(q, cache, bt)
    g = torch.Generator(device="cuda").manual_seed(5)
    for fill in ("ones", "random", "reuse", "reuse"):
        if fill == "ones":
            ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
        elif fill == "random":
            ws = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=g)
        out = pkv.paged_decode(q, cache, bt, cl, sm_scale=w.sm_scale, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), fill


@pytest.mark.parametrize("kind", ["bf16", "u3"])
def test_graph_replays_of_one_call(pkv, kind):
    """One captured paged_decode call replayed with new queries: every replay
    equals an eager call on the same inputs, bit for bit."""
    if kind == "bf16":
        w = W.gqa_bf16(batch=8, ctx_lo=200, ctx_hi=4000, seed=264)
    else:
        w = W.u3_mha(batch=4, ctx_lo=200, ctx_hi=3000, seed=265)
    cache, _ = PL.gpu_run(w, pkv, decode=False)
    q = w.q.cuda().clone()
    bt, cl = w.block_tables.cuda(), w.context_lens.cuda()
    ws = torch.empty(pkv.decode_workspace_bytes(q, cache, bt), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkv.paged_decode(q, cache, bt, cl, sm_scale=w.sm_scale, out=out, workspace=ws)  # warm-up
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            pkv.paged_decode(q, cache, bt, cl, sm_scale=w.sm_scale, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.Generator(device="cuda").manual_seed(7)
    for _ in range(4):
        q.copy_(torch.randn(q.shape, device="cuda", generator=g).to(q.dtype))
        graph.replay()
        eager = pkv.paged_decode(q, cache, bt, cl, sm_scale=w.sm_scale)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
