"""Decode steps captured in a CUDA graph (the pages' remedy for launch
overhead, "Nano-vLLM System Architecture Analysis", §2 "CUDA Graphs").  The
library reads lengths, tables and slots from device memory and allocates
nothing, so one captured step serves every batch of the same shape: change the
inputs in place, replay, and the results equal eager calls."""
import pytest
import torch

from paged_kv_cache_214_gb300 import pkv
from paged_kv_cache_214_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_replayed_graph_matches_eager_after_inputs_change():
    dev = "cuda"
    lens_a = [300, 4000, 1000, 2500, 17, 513, 3333, 4096]
    lens_b = [4096, 12, 2222, 800, 1500, 256, 257, 3000]
    wa = W.make_decode(lens_a, 32, 8, 160, 9000, pool_device=dev, max_blocks_per_seq=16)
    wb = W.make_decode(lens_b, 32, 8, 160, 9001, pool_device=dev, max_blocks_per_seq=16)
    kc, vc = wa.k_cache.clone(), wa.v_cache.clone()
    # static input buffers the graph reads
    q = wa.q.to(dev).clone()
    kn, vn = wa.k_new.to(dev).clone(), wa.v_new.to(dev).clone()
    slots = wa.slot_mapping.to(dev).clone()
    tables = wa.block_tables.to(dev).clone()
    lens = wa.context_lens.to(dev).clone()
    out = torch.empty_like(q)
    lse = torch.empty((wa.B, wa.Hq), dtype=torch.float32, device=dev)
    need = pkv.paged_decode_workspace_bytes(wa.B, wa.Hq, wa.Hkv, wa.D, 16)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)

    def step(stream):
        pkv.kv_cache_store(kn, vn, kc, vc, slots, stream=stream)
        pkv.paged_decode_attention(q, kc, vc, tables, lens, wa.scale, out=out, lse=lse,
                                   workspace=ws, stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s)                       # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    torch.cuda.synchronize()

    for w in (wa, wb, wa):
        kc_e, vc_e = kc.clone(), vc.clone()
        q.copy_(w.q)
        kn.copy_(w.k_new)
        vn.copy_(w.v_new)
        slots.copy_(w.slot_mapping)
        tables.copy_(w.block_tables)
        lens.copy_(w.context_lens)
        g.replay()
        torch.cuda.synchronize()
        o_graph, l_graph = out.clone(), lse.clone()
        # eager on a copy of the pool as it was before the replay
        pkv.kv_cache_store(kn, vn, kc_e, vc_e, slots)
        o_e, l_e = pkv.paged_decode_attention(q, kc_e, vc_e, tables, lens, w.scale)
        torch.cuda.synchronize()
        assert torch.equal(kc, kc_e) and torch.equal(vc, vc_e)
        assert torch.equal(o_graph, o_e) and torch.equal(l_graph, l_e)
    assert pkv.get_device_error() == pkv.PKV_OK
