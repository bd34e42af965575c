"""GPU parity of top-k Gumbel-max sampling (q4_sample_topk) against the CPU oracle
(oracle/sampler_oracle.py): the ranked top-k indices and the token must be identical.

The rumik-oss-1 write-up samples on the GPU ("Step 4": top-k with the Gumbel-max trick; "Steps
9-10": top-k by sorting 64-bit keys of float bits and index).  Both sides get the same float32
noise and score in the same float32 arithmetic, so every decision is taken in the same precision.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle.sampler_oracle as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int4_weight_only_q4_gb300 as m
    return m


def run(q4, y, k, invt, noise, offset=0):
    flat = np.zeros(y.size + offset, np.float32)
    flat[offset:] = y.reshape(-1)
    dev = torch.from_numpy(flat).cuda()
    Y = dev[offset:].view(y.shape)                 # offset 1: rows not 16-byte aligned (scalar path)
    tok, idx = q4.sample_topk(Y, k, invt, torch.from_numpy(noise).cuda(), return_topk=True)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), idx.cpu().numpy()


def check(q4, y, k, invt, seed, offset=0):
    rng = np.random.default_rng(seed)
    noise = S.gumbel_noise(np.clip(rng.random((y.shape[0], k)), 1e-12, 1 - 1e-12))
    tok, idx = run(q4, y, k, invt, noise, offset)
    want_t, want_i = S.sample(y, k, invt, noise)
    assert np.array_equal(idx, want_i)
    assert np.array_equal(tok, want_t)


@pytest.mark.parametrize("N,k", [(1, 1), (7, 3), (100, 100), (4097, 50), (65536, 1), (65536, 50), (65536, 1024),
                                 (70001, 64)])
@pytest.mark.parametrize("B", [1, 3, 8])
def test_random_logits(q4, N, k, B):
    rng = np.random.default_rng(N + k + B)
    y = (rng.standard_normal((B, N)) * 3).astype(np.float32)
    check(q4, y, k, 1.0 / 0.8, seed=B)


def test_misaligned_rows_and_temperatures(q4):
    rng = np.random.default_rng(1)
    y = (rng.standard_normal((4, 65536)) * 2).astype(np.float32)
    for invt in (0.25, 1.0, 3.7):
        check(q4, y, 40, invt, seed=int(invt * 10), offset=1)
        check(q4, y, 40, invt, seed=int(invt * 10))


def test_many_ties_at_the_threshold(q4):
    # logits on a coarse grid: thousands of equal values, the k-th value shared by many indices
    rng = np.random.default_rng(2)
    y = np.round(rng.standard_normal((3, 65536)) * 2).astype(np.float32)
    for k in (1, 10, 300, 1024):
        check(q4, y, k, 1.0, seed=k)
    y[1] = 5.0                                      # every logit equal: the first k indices
    check(q4, y, 37, 1.0, seed=9)


def test_special_values(q4):
    y = np.random.default_rng(3).standard_normal((4, 5000)).astype(np.float32)
    y[0, [10, 4000]] = np.nan                       # NaN ranks first, lower index first
    y[1, :] = -np.inf
    y[1, 77] = -1e30
    y[2, ::2] = -0.0
    y[2, 1::2] = 0.0                                # -0 and +0 are equal values
    y[3, 123] = np.inf
    for k in (1, 5, 64):
        check(q4, y, k, 1.0, seed=k)


def test_greedy_cases_match_argmax(q4):
    rng = np.random.default_rng(4)
    y = rng.standard_normal((8, 65536)).astype(np.float32)
    Y = torch.from_numpy(y).cuda()
    zero = torch.zeros((8, 16), device="cuda")
    tok = q4.sample_topk(Y, 16, 1.0, zero)
    am = q4.argmax(Y)
    torch.cuda.synchronize()
    assert torch.equal(tok, am)


@pytest.mark.parametrize("cluster", ["1", "0"])
def test_each_kernel_on_every_candidate_path(q4, monkeypatch, cluster):
    """k <= 128 runs one cluster of CTAs per row (Q4_SAMPLE_CLUSTER=0 forces the one-CTA kernel):
    rows whose chunks gather few candidates (ranked by counting), hundreds (a bitonic sort) or more
    than fit (the exact radix select with ordered ties), empty chunks of short rows, and rows that
    do not start on a 16-byte boundary -- every one equal to the oracle."""
    monkeypatch.setenv("Q4_SAMPLE_CLUSTER", cluster)
    rng = np.random.default_rng(11)
    cases = [
        (rng.standard_normal((2, 65536)) * 3, 50),                      # few candidates per chunk
        (rng.integers(0, 10, (2, 65536)), 50),                          # ~800 equal top values per chunk
        (rng.integers(0, 3, (2, 65536)), 64),                           # more than fit: exact path
        (np.zeros((2, 65536)), 128),                                    # one value everywhere
        (rng.standard_normal((3, 33)), 33),                             # short rows: some chunks empty
        (rng.standard_normal((2, 5)), 2),
        (rng.standard_normal((2, 70001)), 128),                         # N not a multiple of 4
        (np.round(rng.standard_normal((2, 65536)) * 2), 1),
    ]
    for i, (y, k) in enumerate(cases):
        y = np.ascontiguousarray(y, dtype=np.float32)
        check(q4, y, k, 1.25, seed=100 + i)
        check(q4, y, k, 0.5, seed=200 + i, offset=1)
