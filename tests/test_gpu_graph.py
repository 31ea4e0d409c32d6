"""spmm_run inside a CUDA graph: capture, replay, same bits as the eager call.

Every family's launch is a plain kernel launch on the caller's stream (the
tensor maps are encoded on the host and passed by value, the split-row and
open-row workspace is reserved beforehand, BLOCK's diagonal blocks are
prepared by the eager call), so a product can be captured once and
replayed. The replayed results must equal the eager ones bit for bit, and the
eager ones are held to the oracle as in the other parity tests.
"""
import pytest

import gen
from parity_util import compare, make_adj, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdm(cuda_device):
    import sparse_dense_matrix_gb300 as m
    return m


CASES = [
    # (graph, N, reduce, pinned family or None)
    ("knn", 16, "sum", "window"),
    ("knn", 64, "mean", "window"),
    ("rmat", 64, "sum", None),          # WARPROW + the two split-row launches
    ("rmat", 128, "max", None),
    ("er", 32, "max", None),            # ROWGROUP
    ("community", 128, "sum", "block"),
    ("rmat", 16, "sum", "segment"),     # merge-path tiles + the open-row launch
    ("rmat", 16, "max", "segment"),
]
GRAPHS = {
    "knn": lambda: gen.knn_local(20000, 10, 64, seed=31),
    "rmat": lambda: gen.rmat(scale=13, edge_factor=16, seed=32),
    "er": lambda: gen.erdos_renyi(3000, 3000, 8, seed=33),
    "community": lambda: gen.community(16, 256, 0.2, 5, seed=34),
}


@pytest.mark.parametrize("name,N,red,family", CASES)
def test_graph_replay_matches_eager(sdm, cuda_device, name, N, red, family):
    import torch
    g = GRAPHS[name]()
    B = gen.features(g.K, N, seed=N)
    Bd = to_dev(B, cuda_device)
    adj = make_adj(sdm, g, cuda_device)
    if family:
        adj.set_family(family)
        assert adj.describe(N, red)["family_name"] == family
    adj.reserve(N, red)                    # no allocation inside the capture
    C0 = torch.empty((g.M, N), dtype=torch.float32, device=cuda_device)
    A0 = torch.empty((g.M, N), dtype=torch.int32, device=cuda_device) if red == "max" else None
    adj.reduce(Bd, red, out=C0, argmax=A0)
    torch.cuda.synchronize()
    compare(g, B, red, C0.cpu().numpy(), None if A0 is None else A0.cpu().numpy(),
            label=f"eager {name} N={N} {red}")

    C1 = torch.full_like(C0, float("nan"))
    A1 = None if A0 is None else torch.full_like(A0, -7)
    s = torch.cuda.Stream(cuda_device)
    s.wait_stream(torch.cuda.current_stream(cuda_device))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s, capture_error_mode="relaxed"):
        adj.reduce(Bd, red, out=C1, argmax=A1, stream=s)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(C1.view(torch.int32), C0.view(torch.int32))
    if A0 is not None:
        assert torch.equal(A1, A0)
    sdm.spmm_plan_sync(adj.plan)
    adj.close()
