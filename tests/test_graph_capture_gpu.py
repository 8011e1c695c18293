"""A training step (forward + backward through the C ABI) captured into a CUDA
graph and replayed gives the same bits as the same step run eagerly: every
launch, including the kernels the library forks onto its second stream and
joins back, is recorded in the capture, and no call synchronises the host.
Then the replayed step against the CPU oracle."""
import numpy as np
import pytest
import torch

import activation_sparse_transformer_gate_gb300 as tw
import synth
from test_backward_gpu import check_backward, ctl_fields, dh_gemm_of
from twell_testlib import torch_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw._build.build()
    tw.load()


class Step:
    """Static device buffers of one training step and the two ABI calls."""

    def __init__(self, a, w, lam, dh_density):
        self.w, self.lam = w, lam
        T, D, F = w.T, w.D, w.F
        self.d = {k: torch_dev(a[k]) for k in ("x", "Wg", "Wu", "Wd", "bg", "rb", "dy")}
        self.bufs = tw.TwellBuffers(T, F, w.C, w.K, tw.TWELL_BF16, None, train=True,
                                    dense_density=-1.0, dh_density=dh_density)
        self.ws, self.nws = tw.workspace(T, D, F, w.C, w.K, tw.TWELL_BF16, True)
        dev = "cuda"
        self.y = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
        self.dWg = torch.empty((F, D), dtype=torch.float32, device=dev)
        self.dWu = torch.empty_like(self.dWg)
        self.dWd = torch.empty_like(self.dWg)
        self.dbg = torch.empty((F,), dtype=torch.float32, device=dev)

    def run(self):
        d, w = self.d, self.w
        tw.twell_ffn_forward(d["x"], d["Wg"], d["bg"], d["rb"], d["Wu"], d["Wd"], w.D, 1,
                             self.bufs.t, self.y, self.ws, self.nws)
        tw.twell_ffn_backward(d["x"], d["Wg"], d["Wu"], d["Wd"], self.bufs.t, d["dy"], self.lam,
                              w.D, self.dx, self.dWg, self.dbg, self.dWu, self.dWd, self.ws,
                              self.nws)

    def outputs(self):
        return {k: getattr(self, k).clone() for k in ("y", "dx", "dWg", "dWu", "dWd", "dbg")}

    def poison(self):
        for k in ("y", "dx", "dWg", "dWu", "dWd", "dbg"):
            getattr(self, k).fill_(float("nan"))


@pytest.mark.parametrize("dh_density", [1e-9, -1.0], ids=["dh_gemm", "dh_sddmm"])
def test_training_step_graph_replay_matches_eager(dh_density):
    w = synth.Workload("graph", 640, 256, 1024, 128, 8, "bf16", True, -2.33, 81, hot_tokens=2,
                       seq_len=160, hot_bias=1.5, lam=1e-3, train=True)
    a = synth.generate(w)
    st = Step(a, w, w.lam, dh_density)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        st.run()  # eager (also creates the library's second stream on this thread)
    torch.cuda.synchronize()
    ref = st.outputs()
    ctl = st.ws[:32].cpu().numpy().copy()
    assert dh_gemm_of(ctl) == (1 if dh_density > 0 else 0)
    assert ctl_fields(ctl)[1] == 0 and ctl_fields(ctl)[2] >= 1  # sparse regime, overflow rows
    st.poison()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st.run()
    st.poison()  # capture does not execute: the replay must write everything
    g.replay()
    g.replay()  # twice: the step reads only its inputs, so replays repeat
    torch.cuda.synchronize()
    code, _ = tw.twell_get_status(st.bufs.t)
    assert code == 0
    got = st.outputs()
    for k in ref:
        assert torch.equal(got[k], ref[k]), k
    res = {k: v.double().cpu().numpy() for k, v in got.items()}
    check_backward(a, w, res, w.lam)
    assert np.isfinite(res["dWd"]).all()
