"""The entry points under CUDA-graph capture.

A call validates on the host and enqueues one kernel; nothing in it is a
stream operation other than the launch, and the NVFP4 / FP8 scale factor is a
device pointer, so a sequence of calls can be captured once and replayed on
new contents of the same buffers.  Checked: a graph of a fused NVFP4 call
(swizzled SFs), a reduce-scatter call over every rank, a sharded QK norm and
an all-gather FP8 call, all with programmatic dependent launch, replayed on
two different sets of inputs, gives bit for bit what the same calls give
when launched directly.
"""
import numpy as np
import pytest
import torch

import reduce_residual_rmsnorm_gb300 as pkg
from reduce_residual_rmsnorm_gb300 import workloads as wl
from tests.gpu_util import host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__.build()
    return torch.device("cuda:0")


def _buffers(dev):
    g = torch.Generator().manual_seed(21)
    R, T, H = 4, 40, 1024
    b = {
        "parts": torch.empty((R, T, H), dtype=torch.bfloat16, device=dev),
        "res": torch.empty((T, H), dtype=torch.bfloat16, device=dev),
        "gamma": (torch.rand(H, generator=g) + 0.5).to(torch.bfloat16).to(dev),
        "sf": torch.tensor([200.0], dtype=torch.float32, device=dev),
        "add": torch.empty((T, H), dtype=torch.bfloat16, device=dev),
        "shards": torch.empty((8, 24, 320), dtype=torch.bfloat16, device=dev),
        "qw": (torch.rand(8 * 256, generator=g) + 0.5).to(torch.bfloat16).to(dev),
        "kw": (torch.rand(8 * 64, generator=g) + 0.5).to(torch.bfloat16).to(dev),
        "ag": [torch.empty((c, 384 + 128 + 64), dtype=torch.bfloat16, device=dev)
               for _, c in (pkg.rs_token_split(19, 3, r) for r in range(3))],
        "xg": (torch.rand(384, generator=g) + 0.5).to(torch.bfloat16).to(dev),
        "yg": (torch.rand(128, generator=g) + 0.5).to(torch.bfloat16).to(dev),
    }
    outs = {
        "fp4": pkg.new_outputs(3, T, H, dev, sf_layout=pkg.SFLayout.SWIZZLED_128x4),
        "rs_res": torch.empty((T, H), dtype=torch.bfloat16, device=dev),
        "rs_norm": torch.empty((T, H), dtype=torch.bfloat16, device=dev),
        "q": torch.empty((24, 8 * 256), dtype=torch.bfloat16, device=dev),
        "k": torch.empty((24, 8 * 64), dtype=torch.bfloat16, device=dev),
        "ag_out": torch.empty((19, 576), dtype=torch.bfloat16, device=dev),
        "ag_x": torch.empty((19, 384), dtype=torch.bfloat16, device=dev),
        "ag_y": torch.empty((19, 128), dtype=torch.bfloat16, device=dev),
        "ag_q": torch.empty((19, 384), dtype=torch.uint8, device=dev),
        "ag_s": torch.empty((19, 3), dtype=torch.float32, device=dev),
    }
    return b, outs


def _fill(b, seed):
    g = torch.Generator().manual_seed(seed)
    for k in ("parts", "res", "add", "shards"):
        b[k].copy_(torch.randn(b[k].shape, generator=g).to(torch.bfloat16))
    for t in b["ag"]:
        t.copy_(torch.randn(t.shape, generator=g).to(torch.bfloat16))


def _calls(b, o, stream):
    pkg.ts_fused_reduce_norm(3, b["parts"], b["res"], b["gamma"], 1e-6, b["sf"],
                             sf_layout=pkg.SFLayout.SWIZZLED_128x4, launch_with_pdl=True, stream=stream,
                             **o["fp4"])
    pkg.ts_reducescatter_fused_norm(8, b["parts"], -1, b["add"], b["res"], b["gamma"], 1e-6,
                                    residual_out=o["rs_res"], norm_out=o["rs_norm"], launch_with_pdl=True,
                                    stream=stream)
    pkg.ts_qk_norm_sharded(b["shards"], 256, 64, b["qw"], b["kw"], 1e-6, q_out=o["q"], k_out=o["k"],
                           launch_with_pdl=True, stream=stream)
    pkg.ts_allgather_fused_norm(2, b["ag"], 384, 128, 64, b["xg"], b["yg"], 1e-6, 1e-6,
                                allgather_out=o["ag_out"], x_norm_out=o["ag_x"], y_norm_out=o["ag_y"],
                                quant_out=o["ag_q"], scale_out=o["ag_s"], launch_with_pdl=True, stream=stream)


def _snapshot(o):
    out = {}
    for k, v in o.items():
        if isinstance(v, dict):
            for kk, vv in v.items():
                out[f"{k}.{kk}"] = host(vv).copy()
        else:
            out[k] = host(v).copy()
    return out


def test_captured_calls_replay_like_direct_calls(dev):
    b, o = _buffers(dev)
    stream = torch.cuda.Stream(device=dev)
    _fill(b, 1)
    with torch.cuda.stream(stream):
        _calls(b, o, stream)  # warm-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        _calls(b, o, stream)
    torch.cuda.synchronize()
    for seed in (2, 3):
        _fill(b, seed)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            _calls(b, o, stream)
        torch.cuda.synchronize()
        direct = _snapshot(o)
        for k, v in o.items():  # clobber the outputs before the replay
            for t in (v.values() if isinstance(v, dict) else [v]):
                t.view(torch.uint8).fill_(0xA5)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        replayed = _snapshot(o)
        assert direct.keys() == replayed.keys()
        for k in direct:
            assert np.array_equal(direct[k], replayed[k]), (seed, k)


def test_rank_calls_on_concurrent_streams(dev):
    """The R per-rank reduce-scatter calls on R streams forked from one stream
    and joined back, captured in a CUDA graph (the ranks run at the same time,
    as on R GPUs; their calls share inputs and write disjoint slices): the
    replay gives the bits of one launch over every rank's slice."""
    R, T, H = 8, 1000, 7168
    inp = wl.fused_inputs(wl.FusedShape(R=R, T=T, H=H, p_std=0.5), seed=31)
    g = torch.Generator().manual_seed(32)
    add = torch.randn((T, H), generator=g).to(torch.bfloat16).to(dev)
    parts, res, gamma = inp["partials"].to(dev), inp["residual"].to(dev), inp["gamma"].to(dev)
    for rs, form in ((7, 6), (8, 1)):
        whole = pkg.new_outputs(form, T, H, dev)
        pkg.ts_reducescatter_fused_norm(rs, parts, -1, add, res, gamma, 1e-6, **whole)
        torch.cuda.synchronize()
        per = []
        for rank in range(R):
            start, count = pkg.rs_token_split(T, R, rank)
            per.append((rank, start, count, pkg.new_outputs(form, count, H, dev)))
        main = torch.cuda.Stream(device=dev)
        side = [torch.cuda.Stream(device=dev) for _ in range(R)]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=main):
            for s2, (rank, start, count, outs) in zip(side, per):
                s2.wait_stream(main)
                pkg.ts_reducescatter_fused_norm(rs, parts, rank, add[start:start + count],
                                                res[start:start + count], gamma, 1e-6, stream=s2, **outs)
            for s2 in side:
                main.wait_stream(s2)
        for _ in range(2):
            for _, _, _, outs in per:
                for v in outs.values():
                    v.zero_()
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            for rank, start, count, outs in per:
                for k, v in outs.items():
                    assert np.array_equal(host(v), host(whole[k][start:start + count])), (rs, rank, k)


@pytest.mark.parametrize("flag", ["early", "independent"])
def test_rank_chain_with_pdl_flags_in_a_graph(dev, flag):
    """The R per-rank reduce-scatter calls back to back on one stream with
    launch_with_pdl and TS_FLAG_PDL_EARLY_READ or TS_FLAG_PDL_INDEPENDENT
    (rank 0 without it, so that no run of flagged calls spans two replays),
    captured in a CUDA graph together with a kernel that reads every slice's
    outputs after the chain: each replay gives the bits of one launch over every
    rank's slice, and the kernel after the chain sees all of them."""
    R, T, H = 8, 1500, 7168
    inp = wl.fused_inputs(wl.FusedShape(R=R, T=T, H=H, p_std=0.5), seed=33)
    g = torch.Generator().manual_seed(34)
    add = torch.randn((T, H), generator=g).to(torch.bfloat16).to(dev)
    parts, res, gamma = inp["partials"].to(dev), inp["residual"].to(dev), inp["gamma"].to(dev)
    rs, form = 7, 6
    whole = pkg.new_outputs(form, T, H, dev)
    pkg.ts_reducescatter_fused_norm(rs, parts, -1, add, res, gamma, 1e-6, **whole)
    torch.cuda.synchronize()
    per = []
    for rank in range(R):
        start, count = pkg.rs_token_split(T, R, rank)
        per.append((rank, start, count, pkg.new_outputs(form, count, H, dev)))
    gathered = torch.empty((T, H), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def chain():
        for rank, start, count, outs in per:
            on = rank > 0
            pkg.ts_reducescatter_fused_norm(rs, parts, rank, add[start:start + count], res[start:start + count],
                                            gamma, 1e-6, launch_with_pdl=True,
                                            pdl_early_read=on and flag == "early",
                                            pdl_independent=on and flag == "independent", stream=stream, **outs)
        for rank, start, count, outs in per:  # reads every call's codes after the chain
            gathered[start:start + count].copy_(outs["quant_out"])

    with torch.cuda.stream(stream):
        chain()  # warm-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        chain()
    want_codes = host(whole["quant_out"])
    for _ in range(2):
        for _, _, _, outs in per:
            for v in outs.values():
                v.view(torch.uint8).fill_(0xA5)
        gathered.fill_(0x5A)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        for rank, start, count, outs in per:
            for k, v in outs.items():
                assert np.array_equal(host(v), host(whole[k][start:start + count])), (flag, rank, k)
        assert np.array_equal(host(gathered), want_codes), flag
