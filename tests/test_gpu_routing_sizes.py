"""Routing permutation at route counts that cross the routing kernels'
boundaries: one block does the count, scan and scatter for up to 2048 routes
(in 1024-route chunks), three kernels beyond.  The permutation is a stable
counting sort by expert (histogram, prefix scan, scatter; within an expert,
routes in (t, k) order), so the GPU's counts, group offsets, perm and inv must
equal the oracle's bit for bit, whatever path produced them.  Small H and I keep the
forward cheap; only the routing outputs are checked here.
"""
import numpy as np
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W
from oracle import oracle as O

from helpers import TILE_ROWS

pytestmark = pytest.mark.gpu
DEV = "cuda"

# (T, K, E): one block with one chunk, two chunks, exactly 2048 routes with
# E = 384, E = 1024 (the largest); three kernels at 2049, 2400 and 4096 routes
SIZES = [(128, 8, 64), (129, 8, 64), (256, 8, 384), (500, 4, 1024), (2049, 1, 16), (300, 8, 64),
         (512, 8, 384)]


@pytest.mark.parametrize("T,K,E", SIZES, ids=lambda v: str(v))
def test_routing_bit_exact_across_sizes(T, K, E):
    wl = W.Workload(f"route_T{T}_K{K}_E{E}", T, 256, 256, E, K, "relu2")
    ids, wts = W.make_routing(wl)
    ids = ids.clone()
    g = torch.Generator().manual_seed(W.BASE_SEED + 9)
    holes = torch.randperm(T * K, generator=g)[: max(1, T * K // 50)]
    ids.view(-1)[holes] = -1                       # empty slots
    ids.view(-1)[holes[:3]] = E + 5                # invalid ids: ignored and flagged
    w1, w2 = W.make_weights(wl, device=DEV)
    w = M.prepare_weights(w1, w2, wl.act)
    x = W.make_x(wl, device=DEV)
    c, s, sc = M.quantize_tokens(x)
    ws = M.workspace(w, T, K)
    M.forward(w, c, s, sc, ids.to(DEV), wts.to(DEV), ws=ws)
    torch.cuda.synchronize()
    assert M.moe_nvfp4_read_status(ws) == 7        # MOE_ERR_BAD_EXPERT_ID

    o_ids = ids.clone()
    o_ids[(o_ids < 0) | (o_ids >= E)] = -1
    counts_o, perm_o, _ = O.route(o_ids.numpy().astype(np.int32), E)
    L = M.moe_nvfp4_workspace_layout(w.dims, T, K)
    view = lambda n, dt, shape: M.ws_view(ws, L, n, dt, shape).cpu().numpy()
    counts = view("counts", torch.int32, (E,))
    assert np.array_equal(counts, counts_o)
    tiles = np.ceil(counts / TILE_ROWS).astype(np.int64)
    row0 = view("group_row0", torch.int32, (E,))
    assert np.array_equal(row0, TILE_ROWS * np.concatenate([[0], np.cumsum(tiles)[:-1]]))
    status = view("status", torch.int32, (16,))
    assert status[1] == tiles.sum() and status[3] == min(TILE_ROWS, counts.max())
    start = np.concatenate([[0], np.cumsum(counts)[:-1]])
    q_expert = np.repeat(np.arange(E), counts)
    rmap = row0[q_expert] + (np.arange(counts.sum()) - start[q_expert])
    perm = view("perm", torch.int32, (L["rows_cap"],))
    assert np.array_equal(perm[rmap], perm_o)
    want = np.full(T * K, -1, np.int64)
    want[perm_o] = rmap
    assert np.array_equal(view("inv", torch.int32, (T * K,)), want)
