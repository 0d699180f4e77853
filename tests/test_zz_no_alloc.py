"""gdn_segmented_fwd_noalloc: the segmented forward for callers that cannot allocate device
memory (a framework that owns all device memory through its own pool, a request path that
must not pay an allocation's implicit synchronisation, a program holding only imported
buffers). It takes its scratch from a fixed array inside the library instead of a caller
workspace. Here it is called through the C ABI and compared with gdn_segmented_fwd and with the
fp64 oracle, twice in a row (the array keeps the previous call's contents, so the second call
must not be disturbed by the first).

This file is named so that pytest collects it last; it passes alone in a fresh process too.
"""
import pytest
import torch

from context_scan_gb300 import gdn, synth
from gpu_util import TOL_BF16, TOL_F32, np64, oracle_ref, rel_err, upload

pytestmark = pytest.mark.gpu

CASES = {
    "cp4_small": (synth.scaled(synth.WORKLOADS["cp4_b2_h32_t32k"], B=2, H=3, T=1024), TOL_BF16),
    "tiny_f32": (synth.WORKLOADS["tiny_f32_k64_cp4"], TOL_F32),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from context_scan_gb300 import _build
    _build.build_cuda()
    gdn.lib()


def _alloc_out(d, w):
    B, T, H, K = d["k"].shape
    return (torch.empty((B, T, H, w.V), device="cuda"),
            torch.empty((B, H, K, w.V), device="cuda"))


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_workspace_entry_point_twice(name):
    w, tol = CASES[name]
    x = synth.make_inputs(w)
    o_or, hf_or, _ = oracle_ref(x, w.seg_len)
    d = upload(x, w)
    o_ref, hf_ref = _alloc_out(d, w)
    prob = gdn.problem(d["k"], d["v"], o_ref)
    ws = gdn.alloc_workspace(prob, w.nseg)
    gdn.gdn_segmented_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o_ref, hf_ref,
                          w.nseg, ws, prob=prob)
    torch.cuda.synchronize()
    err_word = torch.full((2,), 123, dtype=torch.int32, device="cuda")
    for call in range(2):
        o, hf = _alloc_out(d, w)
        o.fill_(float("nan"))
        gdn.gdn_segmented_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, hf,
                                      w.nseg, device_error=err_word, prob=prob)
        torch.cuda.synchronize()
        assert err_word.tolist() == [0, 0], (call, err_word.tolist())
        assert rel_err(np64(o), np64(o_ref)) <= tol, call
        assert rel_err(np64(hf), np64(hf_ref)) <= tol, call
        assert rel_err(np64(o), o_or, label="o vs oracle") <= tol, call
        assert rel_err(np64(hf), hf_or, label="h_final vs oracle") <= tol, call


def test_noalloc_rejects_problems_beyond_the_array():
    # B*H = 512 heads of 256 tokens in 2 segments (2 pieces) need 512*(4*10 KiB) of WY tiles
    # and 2*512*64 KiB of piece states: more than the fixed array
    w = synth.scaled(synth.WORKLOADS["cp2_b16_h32_t4k"], T=256)
    d = {n: torch.zeros((w.B, w.T, w.H, w.K), dtype=torch.bfloat16, device="cuda")
         for n in ("q", "k", "v")}
    d["g"] = torch.zeros((w.B, w.T, w.H), dtype=torch.bfloat16, device="cuda")
    d["beta"] = torch.zeros((w.B, w.T, w.H), dtype=torch.bfloat16, device="cuda")
    o = torch.full((w.B, w.T, w.H, w.V), 5.0, device="cuda")
    hf = torch.empty((w.B, w.H, w.K, w.V), device="cuda")
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_segmented_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], None, o, hf,
                                      w.nseg)
    assert e.value.status == 5
    torch.cuda.synchronize()
    assert (o == 5.0).all()
