"""GPU parity of the tensor-core paged prefill attention (pkv_prefill_attention) against the oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_kv_cache_88_gb300 as pkv  # noqa: E402
from oracle import ref_attn as rf  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


def _case(lens, chunks, H, B, seed, nan_canary=True):
    D = 128
    rng = np.random.default_rng(seed)
    nb = [-(-t // B) for t in lens]
    N = sum(nb) + 3
    perm = rng.permutation(N)
    tables = np.zeros((len(lens), max(nb)), dtype=np.int32)
    i = 0
    for s, n in enumerate(nb):
        tables[s, :n] = perm[i:i + n]
        i += n
    kp = rng.standard_normal((N, H, B, D)).astype(np.float16)
    vp = rng.standard_normal((N, H, B, D)).astype(np.float16)
    if nan_canary:   # slots past each sequence's tokens hold NaN
        for s, T in enumerate(lens):
            last = tables[s, nb[s] - 1]
            off = T - (nb[s] - 1) * B
            kp[last, :, off:] = np.float16(np.nan)
            vp[last, :, off:] = np.float16(np.nan)
    q = rng.standard_normal((sum(chunks), H, D)).astype(np.float16)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    return q, q_start, kp, vp, tables, np.asarray(lens, dtype=np.int32), N


def _run(q, q_start, kp, vp, tables, lens, N, H, B, max_chunk, scale=0.0):
    dev = "cuda"
    pool = pkv.Pool(1, N, B, H, 128, "HND", k_pool=torch.from_numpy(kp).to(dev), v_pool=torch.from_numpy(vp).to(dev))
    qd = torch.from_numpy(q).to(dev)
    out = torch.full_like(qd, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pool.prefill_attention(0, qd, torch.from_numpy(q_start).to(dev), max_chunk, torch.from_numpy(tables).to(dev),
                           torch.from_numpy(lens).to(dev), out, status, scale=scale)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), int(status.item())


def _check(got, ref, what):
    err = np.abs(got - ref)
    bad = ~(err <= ATOL + RTOL * np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance, max err {np.nanmax(err):.3e}"


@pytest.mark.parametrize("B", [8, 16, 64, 256, 512])
def test_prefill_mixed_chunks(B):
    H = 2
    lens, chunks = [200, 130, 300, 5], [200, 17, 129, 5]
    q, qs, kp, vp, tab, ln, N = _case(lens, chunks, H, B, seed=B)
    got, st = _run(q, qs, kp, vp, tab, ln, N, H, B, max(chunks))
    assert st == 0
    ref = rf.prefill_attention(q, kp, vp, tab, ln, qs, B, layout="HND")
    _check(got, ref, f"B={B}")


@pytest.mark.parametrize("B", [16, 128])
def test_prefill_tile_pairs(B):
    """Each CTA takes two query tiles: the second may be absent or ragged, and may need the
    same number of key tiles as the first (then the first zeroes the last tile's dead V rows)
    or one more (then the second does); NaN canaries sit past every context."""
    H = 2
    lens, chunks = [190, 140, 400, 256, 257], [180, 140, 390, 256, 129]
    q, qs, kp, vp, tab, ln, N = _case(lens, chunks, H, B, seed=11 + B)
    got, st = _run(q, qs, kp, vp, tab, ln, N, H, B, max(chunks))
    assert st == 0
    ref = rf.prefill_attention(q, kp, vp, tab, ln, qs, B, layout="HND")
    _check(got, ref, f"tile pairs B={B}")


def test_prefill_long_context_several_tiles():
    H, B = 4, 16
    lens, chunks = [2048, 1500, 700], [512, 300, 700]
    q, qs, kp, vp, tab, ln, N = _case(lens, chunks, H, B, seed=7, nan_canary=False)
    got, st = _run(q, qs, kp, vp, tab, ln, N, H, B, 700, scale=0.1)
    assert st == 0
    ref = rf.prefill_attention(q, kp, vp, tab, ln, qs, B, layout="HND", scale=0.1)
    _check(got, ref, "long context")


def test_prefill_single_token_chunks_match_decode():
    """A chunk of one token is a decode step: both kernels agree with the oracle."""
    H, B = 2, 16
    lens, chunks = [1, 33, 257], [1, 1, 1]
    q, qs, kp, vp, tab, ln, N = _case(lens, chunks, H, B, seed=3)
    got, st = _run(q, qs, kp, vp, tab, ln, N, H, B, 1)
    assert st == 0
    ref = rf.decode_attention(q, kp, vp, tab, ln, B, layout="HND")
    _check(got, ref, "single-token chunks")


def test_prefill_rejects_other_pools():
    pool = pkv.Pool(1, 4, 16, 2, 64, "HND", k_pool=torch.zeros(4 * 16 * 2 * 64, dtype=torch.float16, device="cuda"),
                    v_pool=torch.zeros(4 * 16 * 2 * 64, dtype=torch.float16, device="cuda"))
    z = torch.zeros((1, 2, 64), dtype=torch.float16, device="cuda")
    i = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pool.prefill_attention(0, z, i, 1, torch.zeros((1, 1), dtype=torch.int32, device="cuda"),
                               torch.ones(1, dtype=torch.int32, device="cuda"), z, torch.zeros(1, dtype=torch.int32,
                                                                                              device="cuda"))
    assert e.value.code == "UNSUPPORTED"


def test_prefill_flags_chunk_beyond_max_chunk():
    """max_chunk sizes the grid: a chunk longer than the grid covers is flagged, and the
    rows the grid does cover are still right."""
    H, B = 2, 16
    lens, chunks = [300, 100], [300, 100]
    q, qs, kp, vp, tab, ln, N = _case(lens, chunks, H, B, seed=5)
    got, st = _run(q, qs, kp, vp, tab, ln, N, H, B, max_chunk=200)     # grid covers 256 rows a chunk
    assert st & pkv.DEV_BAD_LENGTH
    ref = rf.prefill_attention(q, kp, vp, tab, ln, qs, B, layout="HND")
    covered = np.r_[0:256, 300:400]
    _check(got[covered], ref[covered], "covered rows")
    got, st = _run(q, qs, kp, vp, tab, ln, N, H, B, max_chunk=300)     # the true bound: no flag
    assert st == 0
    _check(got, ref, "all rows")
