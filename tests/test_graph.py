"""The hot path inside a CUDA graph.

A causal GQA prefill with more units than SMs (the persistent kernel and its
packed schedule) and a split-KV decode with its merge in the split launch are
captured once into a CUDA graph and replayed on new inputs copied into the
captured buffers; every output is compared with the fp64 oracle, and the
decode's completion counters are zero after each replay.  A first call outside
the capture sets up what the library builds once (the error word, the
schedule of the prefill's launch shape, the shared state of the kernels)."""
import pytest
import torch

import oracle
from attention_forward_tcgen05_gb300 import decode, prefill, sync_check
from attention_forward_tcgen05_gb300 import workloads as W
from tests.tolerances import check_lse, check_o

pytestmark = pytest.mark.gpu


def test_prefill_and_decode_replayed_from_a_cuda_graph():
    B, Hq, Hkv, S, d = 1, 28, 4, 1500, 128  # ceil(1500 / 256) * 28 = 168 units > 152 SMs
    lens_h = torch.tensor([1641, 700, 0, 33], dtype=torch.int32)
    Hq_d, Hkv_d, n_splits = 28, 4, 8
    scale = 1.0 / d ** 0.5

    def prefill_inputs(seed):
        return W.prefill_inputs(B, Hq, Hkv, S, S, d, seed)

    def decode_inputs(seed):
        return W.decode_inputs(len(lens_h), Hq_d, Hkv_d, d, lens_h, seed)

    q, k, v = [t.cuda() for t in prefill_inputs(900)]
    o = torch.empty((B, S, Hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    qd, kc, vc = [t.cuda() for t in decode_inputs(901)]
    lens = lens_h.cuda()
    od = torch.empty((len(lens_h), Hq_d, d), dtype=torch.bfloat16, device="cuda")
    ld = torch.empty((len(lens_h), Hq_d), dtype=torch.float32, device="cuda")
    po = torch.empty((len(lens_h), Hq_d, n_splits, d), dtype=torch.float32, device="cuda")
    pl = torch.empty((len(lens_h), Hq_d, n_splits), dtype=torch.float32, device="cuda")
    ctr = torch.zeros(len(lens_h) * Hq_d, dtype=torch.int32, device="cuda")

    def step():
        prefill(q, k, v, causal=True, scale=scale, out=(o, lse))
        decode(qd, kc, vc, lens, n_splits, 1, scale, torch.bfloat16, out=(od, ld), parts=(po, pl), counters=ctr)

    step()  # outside the capture: what the library sets up on first use
    sync_check()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()

    for seed in (910, 920):
        hq, hk, hv = prefill_inputs(seed)
        dq, dk, dv = decode_inputs(seed + 1)
        for dst, src in ((q, hq), (k, hk), (v, hv), (qd, dq), (kc, dk), (vc, dv)):
            dst.copy_(src)
        graph.replay()
        sync_check()
        ro, rl = oracle.sdpa(hq, hk, hv, True, scale)
        check_o(o.float().cpu().numpy(), ro, True, f"graph replay {seed}: prefill O")
        check_lse(lse.cpu().numpy(), rl, f"graph replay {seed}: prefill LSE")
        rdo, rdl = oracle.decode(dq, dk, dv, lens_h, scale)
        check_o(od.float().cpu().numpy(), rdo, True, f"graph replay {seed}: decode O")
        check_lse(ld.cpu().numpy(), rdl, f"graph replay {seed}: decode LSE")
        assert not torch.any(ctr).item(), "completion counters not reset"
