"""The products inside a captured CUDA graph: the six products of a step (the
misaligned ones over the attached transposes) and a normalized view are
captured once and replayed; the replays equal the eager results bit for bit,
including after the dense operands change in place."""
import torch

import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import build as vs_build
from sparse_dense_products_gb300 import workloads as W

import pytest

from gpu_helpers import build

pytestmark = pytest.mark.gpu

STEP = [("vcs", "row", "A@B"), ("vcs", "col", "A@B"), ("vcs", "row", "B@A"),
        ("vcs", "col", "B@A"), ("csr", "row", "A@B"), ("csr", "row", "B@A")]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; none is visible"
    vs_build.build()


def test_step_replays_in_a_cuda_graph():
    coo = W.random_coo(3000, 1200, 150_000, seed=51, values="counts", sort=False)
    H = {}
    for layout, major in {(l, m) for l, m, _ in STEP}:
        H[(layout, major)] = build(coo, layout, major).attach_transpose()
    Xab = W.dense(coo.n_cols, 16, seed=1).cuda()
    Xba = W.dense(coo.n_rows, 16, seed=2).cuda()
    r = (0.5 + torch.rand(coo.n_rows, generator=torch.Generator().manual_seed(4))).cuda()
    outs = [vs.empty_out(H[(l, m)], 16, d) for l, m, d in STEP]
    view_out = vs.empty_out(H[("vcs", "row")], 16, "A@B")

    def step():
        for (l, m, d), o in zip(STEP, outs):
            vs.spmm(H[(l, m)], Xab if d == "A@B" else Xba.t(), d, out=o)
        vs.spmm(H[("vcs", "row")], Xab, "A@B", out=view_out, map="log1p", row_scale=r)

    step()                      # eager: sizes scratch and caches launch parameters
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs] + [view_out.clone()]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for o in outs + [view_out]:
        o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for k, (o, e) in enumerate(zip(outs + [view_out], eager)):
        assert torch.equal(o, e), f"replay differs from eager for product {k}"
    # new operand values, same buffers: the replay computes the new products
    Xab.mul_(-0.5)
    Xba.add_(1.0)
    g.replay()
    torch.cuda.synchronize()
    got = [o.clone() for o in outs] + [view_out.clone()]
    step()
    torch.cuda.synchronize()
    for k, (o, e) in enumerate(zip(got, outs + [view_out])):
        assert torch.equal(o, e), f"replay after an operand change differs for product {k}"
    for h in H.values():
        h.destroy()


def test_wide_matrix_products_replay_in_a_cuda_graph():
    """A matrix with 64-bit slice pointers runs one gather per segment: the
    launches of all segments capture and replay like one product's."""
    coo = W.random_coo(3000, 1200, 150_000, seed=52, values="counts", sort=False)
    c = coo.to("cuda")
    A = vs.build_vcs(c.rows, c.cols, c.vals, (coo.n_rows, coo.n_cols), "row", pointer_bits=64,
                     segment_entries=20_000).attach_transpose()
    assert A.info()["n_segments"] > 5
    Xab = W.dense(coo.n_cols, 16, seed=3).cuda()
    Xba = W.dense(coo.n_rows, 16, seed=4).cuda()
    outs = [vs.empty_out(A, 16, "A@B"), vs.empty_out(A, 16, "B@A")]

    def step():
        vs.spmm(A, Xab, "A@B", out=outs[0])
        vs.spmm(A, Xba.t(), "B@A", out=outs[1])

    step()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for o, e in zip(outs, eager):
        assert torch.equal(o, e)
    A.destroy()
