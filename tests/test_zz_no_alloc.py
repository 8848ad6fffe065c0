"""The allocation-free attention entry point (pkv_decode_attention_static).

Some callers cannot allocate device memory -- a host framework that owns every
device byte and gives a plugin no workspace, or a serving loop that forbids
allocation once it runs. For them the library keeps the attention scratch in a
fixed 4 MiB array of its own. These tests call that entry point through the C
ABI and check its output against pkv_decode_attention (caller workspace), within
the attention tolerance, on two calls in a row (the array keeps the previous
call's contents). The file sorts last so that a run stopping at the first
failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_kv_cache_88_gb300 as pkv  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


def _case(lens, H, D, B, seed):
    rng = np.random.default_rng(seed)
    nb = [-(-t // B) for t in lens]
    N = sum(nb) + 3
    perm = rng.permutation(N)
    tables = np.zeros((len(lens), max(nb)), dtype=np.int32)
    i = 0
    for s, n in enumerate(nb):
        tables[s, :n] = perm[i:i + n]
        i += n
    dev = "cuda"
    q = torch.from_numpy(rng.standard_normal((len(lens), H, D)).astype(np.float16)).to(dev)
    k = torch.from_numpy(rng.standard_normal((N, H, B, D)).astype(np.float16)).to(dev)
    v = torch.from_numpy(rng.standard_normal((N, H, B, D)).astype(np.float16)).to(dev)
    return q, k, v, torch.from_numpy(tables).to(dev), torch.tensor(lens, dtype=torch.int32, device=dev), N


def _static_call(q, k, v, tables, lens, N, B, out, status):
    S, H, D = q.shape
    return pkv.lib().pkv_decode_attention_static(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), N, B, H, D, pkv.LAYOUTS["HND"], tables.data_ptr(),
        tables.shape[1], lens.data_ptr(), S, ctypes.c_float(0.0), out.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("lens,H,D,B", [
    ([17, 300, 1, 64, 1000, 257, 33, 512], 8, 128, 16),   # mixed lengths, several CTAs per sequence
    ([20000], 2, 128, 256),                                # one long sequence split over every CTA
    ([5, 77, 129], 4, 64, 8),
])
def test_static_scratch_matches_workspace_entry_point(lens, H, D, B):
    q, k, v, tables, ln, N = _case(lens, H, D, B, seed=len(lens) + D)
    ref = pkv.decode_attention(q, k, v, tables, ln, num_blocks=N, block_size=B, layout="HND")
    torch.cuda.synchronize()
    r = ref.cpu().numpy().astype(np.float64)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = _static_call(q, k, v, tables, ln, N, B, out, status)
        assert rc == 0, pkv.last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - r) <= ATOL + RTOL * np.abs(r)), f"call {call}: max err {np.abs(got - r).max()}"


def test_static_scratch_rejects_sizes_beyond_its_capacity():
    q = torch.zeros((8, 1, 128), dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tables = torch.zeros((8, 1), dtype=torch.int32, device="cuda")
    lens = torch.ones(8, dtype=torch.int32, device="cuda")
    # 4096 sequences x 256 heads need 4 MiB of counters alone: refused before any launch
    rc = pkv.lib().pkv_decode_attention_static(
        q.data_ptr(), q.data_ptr(), q.data_ptr(), 1, 16, 256, 128, pkv.LAYOUTS["HND"], tables.data_ptr(), 1,
        lens.data_ptr(), 4096, ctypes.c_float(0.0), out.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == 1 and "static scratch holds" in pkv.last_error()
