"""spmm_wcsr_run_noalloc: the WCSR product for callers that cannot allocate
device memory when they run it (their memory comes from their own pool, or
cudaMalloc is off limits at that point).  Its work list and partial sums
live in a static device array instead of memory the handle allocates.

Checked through the C ABI on two calls in a row (the static array keeps the
previous call's contents), element by element against the CPU oracle's C
within the bound every parity test uses, |dC| <= 4*2^-8*sum|a*b| + 1e-6, and
against the ordinary entry point (spmm_run on a handle) within the same
bound.  A window_row_ptr that breaks the format's rules is turned away on
the device without touching C.  This file is collected last so that a
failure here comes after every other test."""
import numpy as np
import pytest

import oracle
import spmm_workloads as W
from spmm_testlib import ensure_library, to_device_bits, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()
    import sparse_dense_matrix_bcsr_gb300 as S
    return S


def _case(name):
    rng = np.random.default_rng({"powerlaw": 11, "tiny": 12, "uniform": 13}[name])
    if name == "powerlaw":       # long windows cut between CTAs
        m, k, n = 2000, 5000, 136
        rp, ci = W.powerlaw_pattern(rng, m, k, 1.3, 1, 1500, 300, 0.7)
    elif name == "tiny":         # fewer work items than SMs; N = 8
        m, k, n = 70, 90, 8
        rp, ci = W.bernoulli_pattern(rng, m, k, 0.1)
    else:                        # uniform 1 %, two 256-wide column tiles + tail
        m, k, n = 4096, 4096, 520
        rp, ci = W.bernoulli_pattern(rng, m, k, 0.01)
    vals = W.draw_values(rng, len(ci), "u1", "bf16")
    B = W.dense_bits(rng, (k, n), "u1", "bf16")
    return m, k, n, rp, ci, vals, B


@pytest.mark.parametrize("name,out_t", [("powerlaw", "f32"), ("tiny", "f32"), ("uniform", "bf16")])
def test_noalloc_matches_handle_on_two_calls(S, name, out_t):
    import torch
    m, k, n, rp, ci, vals, B = _case(name)
    h = S.spmm_wcsr_create(m, k, rp, ci, vals, "bf16", out_t)
    try:
        ptr, idx, values = S.spmm_export_format(h)
        dB = to_device_bits(B, "bf16")
        ref = torch.full((m, n), float("nan"), dtype=torch_dtype(out_t), device="cuda")
        S.run_torch(h, dB, ref)
        torch.cuda.synchronize()
        assert S.spmm_check(h, 0) == S.SPMM_OK
    finally:
        S.spmm_destroy(h)
    ref = ref.double().cpu().numpy()
    C_orc, Sabs = oracle.spmm_csr(m, k, rp, ci, vals, oracle.BF16, B)
    bound = 4.0 * 2.0 ** -8 * Sabs + 1e-6
    assert np.all(np.abs(ref - C_orc) <= bound), "spmm_run differs from the oracle"
    d_ptr = torch.from_numpy(ptr).cuda()
    d_idx = torch.from_numpy(np.ascontiguousarray(idx) if len(idx) else np.zeros(1, np.int32)).cuda()
    d_val = torch.from_numpy(np.ascontiguousarray(values).view(np.int16).reshape(-1)).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        C = torch.full((m, n), float("nan"), dtype=torch_dtype(out_t), device="cuda")
        S.spmm_wcsr_run_noalloc(d_ptr.data_ptr(), d_idx.data_ptr(), d_val.data_ptr(), m, k, len(idx),
                                "bf16", out_t, dB.data_ptr(), C.data_ptr(), n, stream)
        torch.cuda.synchronize()
        assert S.spmm_wcsr_noalloc_check(stream) == S.SPMM_OK
        got = C.double().cpu().numpy()
        assert not np.isnan(got).any(), f"call {call}: C not fully written"
        assert np.all(np.abs(got - C_orc) <= bound), f"call {call}: differs from the oracle beyond the bound"
        assert np.all(np.abs(got - ref) <= 2 * bound), f"call {call}: differs from spmm_run beyond the bound"


@pytest.mark.parametrize("defect", ["not_multiple_of_16", "decreasing", "last_not_p_total", "first_not_zero"])
def test_noalloc_turns_away_a_bad_window_row_ptr(S, defect):
    """A window_row_ptr of the right length whose entries break the format
    (entry not a multiple of 16, decreasing, last entry != p_total, first
    entry != 0): the stage-list kernel finds it before any work is listed, so
    C keeps its contents, and a following valid call still works."""
    import torch
    m, k, n, rp, ci, vals, B = _case("tiny")
    h = S.spmm_wcsr_create(m, k, rp, ci, vals, "bf16", "f32")
    try:
        ptr, idx, values = S.spmm_export_format(h)
    finally:
        S.spmm_destroy(h)
    bad = ptr.copy()
    if defect == "not_multiple_of_16":
        bad[1] += 8
    elif defect == "decreasing":
        bad[1], bad[2] = bad[2] + 16, bad[1]
    elif defect == "last_not_p_total":
        bad[-1] -= 16
    else:
        bad[0] = 16
    assert len(bad) == len(ptr)
    d_idx = torch.from_numpy(np.ascontiguousarray(idx)).cuda()
    d_val = torch.from_numpy(np.ascontiguousarray(values).view(np.int16).reshape(-1)).cuda()
    dB = to_device_bits(B, "bf16")
    stream = torch.cuda.current_stream().cuda_stream
    C = torch.full((m, n), 7.0, dtype=torch.float32, device="cuda")
    S.spmm_wcsr_run_noalloc(torch.from_numpy(bad).cuda().data_ptr(), d_idx.data_ptr(), d_val.data_ptr(), m, k,
                            len(idx), "bf16", "f32", dB.data_ptr(), C.data_ptr(), n, stream)
    torch.cuda.synchronize()
    assert S.spmm_wcsr_noalloc_check(stream) == S.SPMM_ERR_DEVICE_CHECK
    assert bool((C == 7.0).all().item()), "C was written although window_row_ptr was rejected"
    d_ptr = torch.from_numpy(ptr).cuda()
    S.spmm_wcsr_run_noalloc(d_ptr.data_ptr(), d_idx.data_ptr(), d_val.data_ptr(), m, k, len(idx), "bf16", "f32",
                            dB.data_ptr(), C.data_ptr(), n, stream)
    torch.cuda.synchronize()
    assert S.spmm_wcsr_noalloc_check(stream) == S.SPMM_OK
    C_orc, Sabs = oracle.spmm_csr(m, k, rp, ci, vals, oracle.BF16, B)
    assert np.all(np.abs(C.double().cpu().numpy() - C_orc) <= 4.0 * 2.0 ** -8 * Sabs + 1e-6)


def test_noalloc_rejects_problems_beyond_its_scratch(S):
    import torch
    B = torch.zeros(8, 8, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(8, 8, dtype=torch.float32, device="cuda")
    ptr = torch.zeros(2, dtype=torch.int64, device="cuda")
    with pytest.raises(S.SpmmError) as e:
        # ceil(m/16) + p_total/64 far above the static limit; nothing is launched
        S.spmm_wcsr_run_noalloc(ptr.data_ptr(), B.data_ptr(), B.data_ptr(), 1 << 30, 8, 1 << 28, "bf16", "f32",
                                B.data_ptr(), C.data_ptr(), 8, 0)
    assert e.value.status == S.SPMM_ERR_UNSUPPORTED
