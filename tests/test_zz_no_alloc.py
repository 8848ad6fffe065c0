"""The allocation-free attention entry point (pkv_decode_attention_static).

Some callers cannot allocate device memory -- a host framework that owns every
device byte and gives a plugin no workspace, or a serving loop that forbids
allocation once it runs (cudaMalloc can synchronise the device). For them the
library keeps the attention scratch in a fixed 4 MiB array of its own. These
tests call that entry point through the C ABI on two calls in a row (the array
keeps the previous call's contents) and check its output against the float64
oracle within the attention tolerance, and against the workspace entry point;
they cover both block layouts, a NULL status word, and bad block ids and
lengths, whose PKV_DEV_* bits must reach the caller's status word. The file
sorts last so that a run stopping at the first failure has run every other test
first.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_kv_cache_88_gb300 as pkv  # noqa: E402
from oracle import ref_attn_c as rc  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


def _case(lens, H, D, B, seed, layout):
    rng = np.random.default_rng(seed)
    nb = [-(-t // B) for t in lens]
    N = sum(nb) + 3
    perm = rng.permutation(N)
    tables = np.zeros((len(lens), max(nb)), dtype=np.int32)
    i = 0
    for s, n in enumerate(nb):
        tables[s, :n] = perm[i:i + n]
        i += n
    shape = (N, H, B, D) if layout == "HND" else (N, B, H, D)
    q = rng.standard_normal((len(lens), H, D)).astype(np.float16)
    k = rng.standard_normal(shape).astype(np.float16)
    v = rng.standard_normal(shape).astype(np.float16)
    return q, k, v, tables, np.asarray(lens, dtype=np.int32), N


def _dev(*arrays):
    return [torch.from_numpy(a).to("cuda") for a in arrays]


def _static_call(q, k, v, tables, lens, N, B, layout, out, status):
    S, H, D = q.shape
    return pkv.lib().pkv_decode_attention_static(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), N, B, H, D, pkv.LAYOUTS[layout], tables.data_ptr(),
        tables.shape[1], lens.data_ptr(), S, ctypes.c_float(0.0), out.data_ptr(),
        None if status is None else status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _assert_close(got, ref, what):
    err = np.abs(got - ref)
    assert np.all(err <= ATOL + RTOL * np.abs(ref)), f"{what}: max err {err.max()}"


@pytest.mark.parametrize("lens,H,D,B,layout", [
    ([17, 300, 1, 64, 1000, 257, 33, 512], 8, 128, 16, "HND"),   # mixed lengths, several CTAs per sequence
    ([17, 300, 1, 64, 1000, 257, 33, 512], 8, 128, 16, "NHD"),
    ([20000], 2, 128, 256, "HND"),                                # one long sequence split over every CTA
    ([5, 77, 129, 0], 4, 64, 8, "NHD"),                           # an empty context among them
])
def test_static_scratch_matches_oracle(lens, H, D, B, layout):
    q, k, v, tab, ln, N = _case(lens, H, D, B, len(lens) + D, layout)
    ref = rc.decode_attention(q, k, v, tab, ln, B, layout)
    qd, kd, vd, td, lnd = _dev(q, k, v, tab, ln)
    wsref = pkv.decode_attention(qd, kd, vd, td, lnd, num_blocks=N, block_size=B, layout=layout)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(qd, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc_ = _static_call(qd, kd, vd, td, lnd, N, B, layout, out, status)
        assert rc_ == 0, pkv.last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = out.cpu().numpy().astype(np.float64)
        _assert_close(got, ref, f"{layout} call {call}")
        # the same kernel with a caller workspace: the same merge order, so the same bits
        assert torch.equal(out, wsref), f"{layout} call {call}: differs from the workspace entry point"


def test_static_scratch_without_a_status_word():
    """status = NULL: the call still runs (its device flags go to the library's own scratch)."""
    q, k, v, tab, ln, N = _case([40, 700, 3], 4, 128, 16, 5, "HND")
    ref = rc.decode_attention(q, k, v, tab, ln, 16, "HND")
    qd, kd, vd, td, lnd = _dev(q, k, v, tab, ln)
    for call in range(2):
        out = torch.full_like(qd, float("nan"))
        assert _static_call(qd, kd, vd, td, lnd, N, 16, "HND", out, None) == 0, pkv.last_error()
        torch.cuda.synchronize()
        _assert_close(out.cpu().numpy().astype(np.float64), ref, f"no status, call {call}")


def test_static_scratch_reports_bad_block_and_length_to_the_caller():
    """A block id outside the pool is clamped by the kernel (no out-of-range read) and flagged,
    a length past the table is clamped and flagged: both bits land in the caller's status word;
    the next clean call reports 0 and is right again."""
    q, k, v, tab, ln, N = _case([40, 20], 2, 128, 16, 7, "HND")
    qd, kd, vd = _dev(q, k, v)
    out = torch.empty_like(qd)
    bad = tab.copy()
    bad[0, 1] = N + 5
    for t_, l_, bit in ((bad, ln, pkv.DEV_BAD_BLOCK), (tab, np.asarray([40, tab.shape[1] * 16 + 7], np.int32),
                                                       pkv.DEV_BAD_LENGTH)):
        td, lnd = _dev(t_, l_)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _static_call(qd, kd, vd, td, lnd, N, 16, "HND", out, status) == 0, pkv.last_error()
        torch.cuda.synchronize()
        assert int(status.item()) & bit
    td, lnd = _dev(tab, ln)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _static_call(qd, kd, vd, td, lnd, N, 16, "HND", out, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _assert_close(out.cpu().numpy().astype(np.float64), rc.decode_attention(q, k, v, tab, ln, 16, "HND"),
                  "after the flagged calls")


def test_static_scratch_rejects_sizes_beyond_its_capacity():
    q = torch.zeros((8, 1, 128), dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tables = torch.zeros((8, 1), dtype=torch.int32, device="cuda")
    lens = torch.ones(8, dtype=torch.int32, device="cuda")
    # 4096 sequences x 256 heads need 4 MiB of counters alone: refused before any launch
    rc_ = pkv.lib().pkv_decode_attention_static(
        q.data_ptr(), q.data_ptr(), q.data_ptr(), 1, 16, 256, 128, pkv.LAYOUTS["HND"], tables.data_ptr(), 1,
        lens.data_ptr(), 4096, ctypes.c_float(0.0), out.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc_ == 1 and "static scratch holds" in pkv.last_error()
