"""A decode step over several layers captured once in a CUDA graph and
replayed: every layer's outputs keep parity with the oracle on every replay.
(The layer kernels are launched with programmatic dependent launch; in a graph
those become programmatic edges.)"""
import pytest
import torch

from helpers import np_state
from hybrid_sparse_attention_gb300 import _lib
from test_gpu_layer import build_tiny, check_step, gpu_prefix_pools, oracle_prefix_pools

pytestmark = pytest.mark.gpu


def test_graph_two_layers_c4_then_c128(oracle_mod):
    layers = []
    for kind in (4, 128):
        st, raw = build_tiny(kind)
        s = np_state(st)
        oracle_prefix_pools(oracle_mod, s, raw, kind)
        g = st.to("cuda")
        gpu_prefix_pools(g, raw, kind)
        B, sh = g.seq_len_in.numel(), g.shape
        res = {"out": torch.empty(B, sh.Hq, sh.Dv, dtype=torch.bfloat16, device="cuda"),
               "lse": torch.empty(B, sh.Hq, dtype=torch.float32, device="cuda"),
               "seq_len_out": torch.empty_like(g.seq_len_in)}
        kw = {}
        if kind == 4:
            res["idx"] = torch.empty(B, sh.k, dtype=torch.int32, device="cuda")
            res["scores"] = torch.zeros(g.kv_pool.shape[0], dtype=torch.float32, device="cuda")
            kw = dict(topk_idx=res["idx"], scores=res["scores"])
        desc = _lib.layer_desc(g, res["out"], res["lse"], res["seq_len_out"], **kw)
        ws = _lib.workspace(_lib.hsa_layer_decode_workspace_size(desc))
        layers.append((kind, g, s, res, desc, ws))
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _, _, _, _, desc, ws in layers:
            _lib.hsa_layer_decode(desc, ws=ws)
    refs = [oracle_mod.layer_decode(s) for _, _, s, _, _, _ in layers]
    for replay in range(2):
        for _, _, _, res, _, _ in layers:
            for t in res.values():
                t.fill_(0)           # a stale output would not pass
        graph.replay()
        torch.cuda.synchronize()
        for (kind, g, s, res, _, ws), ref in zip(layers, refs):
            assert _lib.hsa_workspace_status(ws) == 0
            check_step(oracle_mod, g, s, res, ref, min_agree=62 / 64)
