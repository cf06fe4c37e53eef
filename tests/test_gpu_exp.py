"""The library's own fp32 exponentials against float64 exp and CUDA's expf:
the accurate scalar routine (os_exp_f32) and the per-element exponentials of
the streaming kernel's fp32 results (os_exp_pairs_f32) and bf16 results
(os_exp_pairs_coarse_f32)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

FLT_MIN = float(np.finfo(np.float32).tiny)


@pytest.fixture(scope="module")
def st():
    import softmax_topk_gb300
    return softmax_topk_gb300


def _ulps(got: np.ndarray, want64: np.ndarray) -> np.ndarray:
    ulp = np.spacing(want64.astype(np.float32)).astype(np.float64)
    return np.abs(got.astype(np.float64) - want64) / ulp


def test_error_bound_on_the_softmax_domain(st):
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    z = torch.cat([-torch.rand(1 << 22, generator=g, device="cuda") * 87.33,
                   -torch.rand(1 << 20, generator=g, device="cuda") * 2.0,
                   -torch.rand(1 << 16, generator=g, device="cuda") * 1e-3,
                   torch.linspace(-87.33, 0.0, 1 << 20, device="cuda")])
    got = st.exp(z)
    torch.cuda.synchronize()
    z64 = z.double().cpu().numpy()
    want = np.exp(z64)
    ulps = _ulps(got.cpu().numpy(), want)
    assert ulps.max() <= 2.0, f"max {ulps.max():.3f} ulp at z={z64[np.argmax(ulps)]}"
    cuda = torch.exp(z).cpu().numpy()          # CUDA's expf on the same inputs
    assert _ulps(cuda, want).max() <= 2.0
    diff = np.abs(got.cpu().numpy().astype(np.float64) - cuda) / want
    assert diff.max() <= 3 * 2.0 ** -23


def test_special_values(st):
    z = torch.tensor([0.0, -0.0, -np.inf, -88.0, -87.5, -100.0, -1e30, -87.33, 1.0, 10.0, 88.0],
                     device="cuda")
    got = st.exp(z).cpu().numpy()
    assert got[0] == 1.0 and got[1] == 1.0
    assert got[2] == 0.0 and not np.signbit(got[2])
    assert 0.0 <= got[3] <= FLT_MIN and 0.0 <= got[4] <= FLT_MIN
    assert got[5] == 0.0 and got[6] == 0.0
    assert got[7] >= FLT_MIN
    want = np.exp(np.array([1.0, 10.0, 88.0]))
    assert np.all(_ulps(got[8:], want) <= 2.0)


def test_in_place(st):
    z = -torch.rand(1000, device="cuda") * 50
    ref = st.exp(z)
    st.os_exp_f32(z.data_ptr(), z.data_ptr(), z.numel(), torch.cuda.current_stream().cuda_stream)
    assert torch.equal(z, ref)


def test_pairs_error_bound_on_the_softmax_domain(st):
    """The streaming kernel's exponential: degree-5 fit (1.1e-7) plus the
    rounding of its evaluation, within 3e-7 relative on z in [-87.33, 0]."""
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    z = torch.cat([-torch.rand(1 << 22, generator=g, device="cuda") * 87.33,
                   -torch.rand(1 << 20, generator=g, device="cuda") * 2.0,
                   -torch.rand(1 << 16, generator=g, device="cuda") * 1e-3,
                   torch.linspace(-87.33, 0.0, (1 << 20) + 1, device="cuda")])
    got = st.exp(z, pairs=True)
    torch.cuda.synchronize()
    z64 = z.double().cpu().numpy()
    want = np.exp(z64)
    rel = np.abs(got.cpu().numpy().astype(np.float64) - want) / want
    assert rel.max() <= 3e-7, f"max rel {rel.max():.3e} at z={z64[np.argmax(rel)]}"


def test_pairs_special_values_and_odd_length(st):
    z = torch.tensor([0.0, -0.0, -np.inf, -88.0, -87.5, -100.0, -1e30, -87.33, -1.0],
                     device="cuda")  # odd length: the last value is paired with 0
    got = st.exp(z, pairs=True).cpu().numpy()
    assert got[0] == 1.0 and got[1] == 1.0
    assert got[2] == 0.0 and not np.signbit(got[2])
    assert 0.0 <= got[3] <= FLT_MIN and 0.0 <= got[4] <= FLT_MIN
    # below e^-87.33 the result is 0 or below FLT_MIN (e^-100 is an fp32
    # subnormal; anything under e^-110, -1e30 included, is exactly +0)
    assert 0.0 <= got[5] <= FLT_MIN and got[6] == 0.0 and not np.signbit(got[6])
    assert got[7] >= FLT_MIN
    assert abs(float(got[8]) - np.exp(-1.0)) <= 3e-7 * np.exp(-1.0)
    w = -torch.rand(1001, device="cuda") * 50
    ref = st.exp(w, pairs=True)
    st.os_exp_pairs_f32(w.data_ptr(), w.data_ptr(), w.numel(), torch.cuda.current_stream().cuda_stream)
    assert torch.equal(w, ref)


def test_coarse_pairs_error_bound(st):
    """The bf16 results' exponential: degree-3 fit (1.0e-4) plus rounding,
    within 1.2e-4 relative on z in [-87.33, 0]; special values as the fine
    form."""
    g = torch.Generator(device="cuda")
    g.manual_seed(2)
    z = torch.cat([-torch.rand(1 << 22, generator=g, device="cuda") * 87.33,
                   -torch.rand(1 << 20, generator=g, device="cuda") * 2.0,
                   torch.linspace(-87.33, 0.0, (1 << 20) + 1, device="cuda")])
    got = st.exp(z, pairs=True, coarse=True)
    torch.cuda.synchronize()
    z64 = z.double().cpu().numpy()
    want = np.exp(z64)
    rel = np.abs(got.cpu().numpy().astype(np.float64) - want) / want
    assert rel.max() <= 1.2e-4, f"max rel {rel.max():.3e} at z={z64[np.argmax(rel)]}"
    s = torch.tensor([0.0, -0.0, -np.inf, -88.0, -100.0, -1e30, -87.33], device="cuda")
    out = st.exp(s, pairs=True, coarse=True).cpu().numpy()
    assert out[0] == 1.0 and out[1] == 1.0
    assert out[2] == 0.0 and not np.signbit(out[2]) and out[5] == 0.0
    assert 0.0 <= out[3] <= FLT_MIN and 0.0 <= out[4] <= FLT_MIN and out[6] >= FLT_MIN
