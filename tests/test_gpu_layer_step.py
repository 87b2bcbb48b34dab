"""A model step through several GDN layers captured in one CUDA graph
("flashinfer.gdn_paged", §Page table: one slots call per step serves every
layer; the F1 drill hint, §plan / run: a step whose calls read only device data
can be captured and replayed).  Every layer has its own pool and inputs; each
replay must match the oracle layer by layer and equal the same step run
eagerly bit for bit."""
import numpy as np
import pytest
import torch

import gated_deltanet_paged_gb300 as gdn
import oracle
from gated_deltanet_paged_gb300 import workloads
from conftest import bf16_bits, f32, i32
from gpu_util import SCALE, Errors, bits_equal, check_o, check_pool

pytestmark = pytest.mark.gpu


def _to_cuda(call):
    kw = {f: (getattr(call, f).cuda().contiguous() if isinstance(getattr(call, f), torch.Tensor) else getattr(call, f))
          for f in call.__dataclass_fields__}
    return type(call)(**kw)


def _decode_step(calls, pools, slots, outs):
    c0 = calls[0]
    gdn.gdn_paged_decode_slots(c0.page_indptr, c0.page_indices, c0.last_page_len, out=slots)
    for l, c in enumerate(calls):
        gdn.gdn_gated_delta_rule_decode_paged(c.q, c.k, c.v, c.g, c.beta, pools[l], c.page_indices, c.page_indptr,
                                              c.last_page_len, scale=SCALE, slots=slots, o=outs[l])


def _prefill_step(calls, pools, slots, outs, ws):
    c0 = calls[0]
    gdn.gdn_paged_prefill_slots(c0.cu_seqlens, c0.page_indptr, c0.page_indices, c0.last_page_len, c0.page_size,
                                out=slots)
    for l, c in enumerate(calls):
        gdn.gdn_chunk_gated_delta_rule_paged(c.q, c.k, c.v, c.g, c.beta, c.cu_seqlens, pools[l], c.page_indices,
                                             c.page_indptr, c.page_size, c.last_page_len, scale=SCALE, slots=slots,
                                             o=outs[l], workspace=ws)


def _capture(step):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step()
    return graph


def _oracle_layers(st_cpu, pools_o, kind):
    """Each layer's call in the oracle: (o, written) per layer; pools_o updated."""
    res = []
    for l, c in enumerate(st_cpu.calls):
        if kind == "decode":
            res.append(oracle.gated_delta_rule_decode_paged(
                bf16_bits(c.q), bf16_bits(c.k), bf16_bits(c.v), f32(c.g), f32(c.beta), pools_o[l],
                i32(c.page_indices), i32(c.page_indptr), i32(c.last_page_len), c.page_size, SCALE))
        else:
            res.append(oracle.chunk_gated_delta_rule_paged(
                bf16_bits(c.q), bf16_bits(c.k), bf16_bits(c.v), f32(c.g), f32(c.beta), i32(c.cu_seqlens),
                pools_o[l], i32(c.page_indices), i32(c.page_indptr), c.page_size, i32(c.last_page_len), SCALE))
    return res


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_graph_captured_layer_step(kind):
    L = 3
    if kind == "decode":
        st = workloads.decode_layers("cpu", L=L, B=6, H=2, max_ctx=3000, seed=51, sentinel=True)
    else:
        st = workloads.prefill_layers("cpu", L=L, S=3, T_seq=300, H=2, page_size=128, seed=52, sentinel=True)
    calls = [_to_cuda(c) for c in st.calls]
    c0 = calls[0]
    pools = st.pools.cuda()
    eager_pools = pools.clone()
    H = st.H
    if kind == "decode":
        B = c0.q.shape[0]
        slots = gdn.gdn_paged_decode_slots(c0.page_indptr, c0.page_indices, c0.last_page_len)
        e_slots = {k: v.clone() for k, v in slots.items()}
        outs = [torch.zeros(B, H, 128, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        e_outs = [o.clone() for o in outs]
        step = lambda: _decode_step(calls, pools, slots, outs)
        eager = lambda: _decode_step(calls, eager_pools, e_slots, e_outs)
    else:
        T, S = c0.q.shape[0], c0.cu_seqlens.numel() - 1
        slots = gdn.gdn_paged_prefill_slots(c0.cu_seqlens, c0.page_indptr, c0.page_indices, c0.last_page_len,
                                            c0.page_size)
        e_slots = {k: v.clone() for k, v in slots.items()}
        outs = [torch.zeros(T, H, 128, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        e_outs = [o.clone() for o in outs]
        ws = torch.empty(gdn.gdn_prefill_workspace_bytes(S, T, H), dtype=torch.uint8, device="cuda")
        e_ws = torch.empty_like(ws)
        step = lambda: _prefill_step(calls, pools, slots, outs, ws)
        eager = lambda: _prefill_step(calls, eager_pools, e_slots, e_outs, e_ws)
    torch.cuda.synchronize()
    before = pools.clone()
    graph = _capture(step)          # capturing runs nothing
    torch.cuda.synchronize()
    assert bits_equal(pools, before)
    pools_o = [st.pools[l].numpy().copy() for l in range(L)]
    errs = Errors()
    for rep in range(2):            # the second replay continues from the first one's states
        prev = pools.clone()
        graph.replay()
        eager()
        torch.cuda.synchronize()
        ref = _oracle_layers(st, pools_o, kind)
        for l in range(L):
            check_o(outs[l], ref[l][0], errs)
            check_pool(pools[l], prev[l], pools_o[l], ref[l][1], errs, "layer %d pool" % l)
            assert bits_equal(outs[l], e_outs[l]) and bits_equal(pools[l], eager_pools[l]), "graph != eager"
    print("%s step, %d layers, graph: %r" % (kind, L, errs))
