"""GPU checks of fw_prefill_noalloc, the prefill entry point that allocates
nothing: the chunked prefill's two-segment form takes its workspace from the
library's static device buffer (FW_SCRATCH_BYTES) instead of the stream-ordered
pool.  Its results equal fw_prefill_ex's bit for bit (same kernels, same split),
on two calls in a row through the same buffer; a call whose two-segment form
would not fit is rejected (FW_ERR_SCRATCH) before anything is launched."""
import pytest
import torch

from linear_token_mixer_gb300 import fw
from linear_token_mixer_gb300 import inputs as I

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_token_mixer_gb300 import build as B
    B.build()
    fw.lib()
    torch.cuda.init()


def _gpu(x):
    return {k: (t.to(DEV) if t is not None else None) for k, t in x.items()}


def _call(w, g, noalloc, o=None, S_T=None):
    o = torch.empty_like(g["q"]) if o is None else o
    S_T = torch.empty(w.B, w.H, w.d, w.d, device=DEV) if S_T is None else S_T
    fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], mode=w.mode, phi=w.phi,
               eps=w.eps, o=o, S_T=S_T, noalloc=noalloc)
    fw.check()
    return o, S_T


@pytest.mark.parametrize("name,shape,split", [
    ("falcon1_bf16", dict(B=2, H=3, T=700), 1),     # two segments forced: the static buffer
    ("linattn_bf16", dict(B=1, H=4, T=333), 1),
    ("falcon1_bf16", dict(B=1, H=2, T=200), 0),     # one segment: no workspace at all
    ("falcon1_long", dict(B=1, H=4, T=4200), 0),    # few long chains: the launch splits by itself
])
def test_noalloc_matches_prefill_ex_on_two_calls(name, shape, split):
    L = fw.lib()
    w = I.WORKLOADS[name].with_shape(**shape)
    g = _gpu(I.prefill_inputs(w, seed=31))
    L.fw_debug_segment_split(split)
    try:
        o_ref, S_ref = _call(w, g, noalloc=False)
        o1, S1 = _call(w, g, noalloc=True)
        o2, S2 = _call(w, g, noalloc=True)   # the same buffer again
    finally:
        L.fw_debug_segment_split(0)
    for o, S in ((o1, S1), (o2, S2)):
        assert torch.equal(o, o_ref)
        assert torch.equal(S, S_ref)


def test_noalloc_rejects_a_split_larger_than_the_buffer():
    """Six chains of 200,000 tokens split into two segments would need
    6 x 100,000 x 256 B of transition outputs (153.6 MB) plus the states, more
    than FW_SCRATCH_BYTES (144 MiB): FW_ERR_SCRATCH, and the outputs stay as
    they were."""
    w = I.WORKLOADS["falcon1_bf16"].with_shape(B=1, H=6, T=200000)
    g = I.prefill_inputs(w, seed=32, device=DEV)
    o = torch.full_like(g["q"], 7.0)
    S_T = torch.full((w.B, w.H, w.d, w.d), 7.0, device=DEV)
    with pytest.raises(fw.FwError) as ei:
        fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], mode=w.mode, phi=w.phi,
                   eps=w.eps, o=o, S_T=S_T, noalloc=True)
    assert ei.value.status == -11
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((S_T == 7.0).all())
    fw.check()   # nothing was launched, so no device error either
