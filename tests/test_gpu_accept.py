"""GPU parity of greedy acceptance and commit (q3kv_accept_greedy) against
oracle/accept.py: accepted counts, next tokens and committed lengths are
integers and must match exactly.  Inputs: seeded synthetic logits from
q3kv_inputs (float32 or bf16-rounded; the oracle gets the exact values the
kernel reads), drafts planted along the oracle's argmax chain for a chosen
number of steps, then a wrong token.
"""
import dataclasses

import numpy as np
import pytest
import torch

import q3kv_inputs as qi
from gpu_harness import GpuCache, check_close, oracle_verify, slot_kv
from oracle.accept import greedy_accept

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _plant(logits, offs, nq, keep, seed, vocab):
    """Query tokens: t_0 random, then `keep[b]` drafts equal to the argmax chain, then wrong ones."""
    toks = qi.random_tokens(seed, logits.shape[0], vocab)
    g = logits.argmax(axis=1)
    for b, T in enumerate(nq):
        r0 = offs[b]
        for j in range(1, T):
            toks[r0 + j] = g[r0 + j - 1] if j <= keep[b] else (g[r0 + j - 1] + 1 + j) % vocab
    return toks


def _run(logits_np, offs, nq, toks, ctx, bf16, max_nq=None, inplace=False):
    from speculative_verify_attention_q3kv_gb300 import api
    rows, vocab = logits_np.shape
    lg = torch.from_numpy(logits_np).cuda()
    if bf16:
        lg = lg.to(torch.bfloat16)
    i32 = dict(dtype=torch.int32, device="cuda")
    S = len(nq)
    ctx_d = torch.tensor(np.asarray(ctx, np.int32), **i32)
    n_acc = torch.full((S,), -7, **i32)
    nxt = torch.full((S,), -7, **i32)
    com = ctx_d if inplace else torch.full((S,), -7, **i32)
    ws = torch.empty(max(api.accept_workspace_bytes(rows, vocab), 8), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, **i32)
    api.accept_greedy(lg, torch.tensor(np.asarray(offs, np.int32), **i32), torch.tensor(np.asarray(nq, np.int32), **i32),
                      torch.tensor(np.asarray(toks, np.int32), **i32), max(nq) if max_nq is None else max_nq,
                      ctx_d, n_acc, nxt, com, ws, st)
    torch.cuda.synchronize()
    return n_acc.cpu().numpy(), nxt.cpu().numpy(), com.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("vocab", [1000, 4099, 50_257, qi.VOCAB])
@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("kind", ["normal", "ties"])
def test_accept_matches_oracle(vocab, bf16, kind):
    rng = np.random.default_rng(vocab + 7 * bf16)
    nq = [int(x) for x in rng.integers(0, 17, size=7)]
    nq[2] = 0                                           # an empty slot
    nq[0] = 16                                          # the widest verify
    offs = np.concatenate([[0], np.cumsum(nq)[:-1]]).astype(np.int32)
    rows = int(sum(nq))
    logits = qi.logits_rows(vocab, rows, vocab, kind, bf16)
    keep = [int(rng.integers(0, max(T, 1))) for T in nq]
    keep[0] = 15                                        # every draft of slot 0 accepted
    toks = _plant(logits, offs, nq, keep, vocab, vocab)
    ctx = [int(x) for x in rng.integers(20, 5000, size=7)]
    want = greedy_accept(logits.astype(np.float64), offs, nq, toks, ctx)
    got = _run(logits, offs, nq, toks, ctx, bf16)
    assert got[3] == 0
    for w_, g_ in zip(want, got[:3]):
        assert np.array_equal(w_, g_), (w_, g_)


def test_accept_in_place_commit_and_status():
    vocab = 3000
    nq = [6, 3]
    offs = [0, 6]
    logits = qi.logits_rows(1, 9, vocab)
    toks = _plant(logits, offs, nq, [2, 1], 1, vocab)
    ctx = [40, 9]
    want = greedy_accept(logits.astype(np.float64), offs, nq, toks, ctx)
    n_acc, nxt, com, st = _run(logits, offs, nq, toks, ctx, False, inplace=True)
    assert st == 0
    assert np.array_equal(n_acc, want[0]) and np.array_equal(nxt, want[1]) and np.array_equal(com, want[2])
    # more query tokens than the launch bound: BAD_LENGTH, the slot keeps its length
    n_acc, nxt, com, st = _run(logits, offs, nq, toks, ctx, False, max_nq=4)
    assert st & 8
    assert (n_acc[0], nxt[0], com[0]) == (0, -1, 40)
    assert (n_acc[1], nxt[1], com[1]) == (want[0][1], want[1][1], want[2][1])
    # a NaN logit is flagged
    bad = logits.copy()
    bad[7, 11] = np.nan
    st = _run(bad, offs, nq, toks, ctx, False)[3]
    assert st & 1


def test_step_accept_commit_then_next_step_overwrites_rejected_rows():
    """Verify step 1 (t_0 + 5 drafts), accept 2 drafts, commit; step 2 appends its
    tokens at the committed length over the rejected rows and verifies: the
    result equals the oracle over the accepted sequence only."""
    w = dataclasses.replace(qi.WORKLOADS[1], num_slots=1, name="accept-e2e")
    c = GpuCache(w, [400], num_layers=1)
    n0, T = 300, 6
    k, v = slot_kv(w, 0, 0, 0, n0 + T)
    c.append_rows(0, [0], [0], [(k, v)])                          # context + t_0 + 5 drafts
    q1 = qi.q_rows(w, 0, 0, 0, T)
    check_close(c.verify(0, [n0 + T], [T], [q1], impl=2), oracle_verify(w, 0, 0, n0, q1, k, v))
    vocab = 5000
    logits = qi.logits_rows(3, T, vocab)
    toks = _plant(logits, [0], [T], [2], 3, vocab)
    n_acc, nxt, com, st = _run(logits, [0], [T], toks, [n0 + T], False)
    assert st == 0 and n_acc[0] == 2 and com[0] == n0 + 3
    # step 2: next token + 4 new drafts appended at the committed length
    rng = np.random.default_rng(5)
    T2 = 5
    k2 = rng.standard_normal((T2, 2, 256)).astype(np.float32)
    v2 = rng.standard_normal((T2, 2, 256)).astype(np.float32)
    c.append_rows(0, [0], [int(com[0])], [(k2, v2)])
    kk = np.concatenate([k[: int(com[0])], k2])
    vv = np.concatenate([v[: int(com[0])], v2])
    q2 = qi.q_rows(w, 0, 0, 1, T2)
    out = c.verify(0, [int(com[0]) + T2], [T2], [q2], impl=2)
    check_close(out, oracle_verify(w, 0, 0, int(com[0]), q2, kk, vv))


# ----------------------------------------------------------------------------- sampled acceptance
from oracle.accept import gumbel_keys, sample_accept, target_prob


def _run_sample(logits_np, offs, nq, toks, ctx, bf16, tau, u, seed):
    from speculative_verify_attention_q3kv_gb300 import api
    rows, vocab = logits_np.shape
    lg = torch.from_numpy(logits_np).cuda()
    if bf16:
        lg = lg.to(torch.bfloat16)
    i32 = dict(dtype=torch.int32, device="cuda")
    S = len(nq)
    out = [torch.full((S,), -7, **i32) for _ in range(3)]
    ws = torch.empty(max(api.accept_workspace_bytes(rows, vocab), 8), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, **i32)
    api.accept_sample(lg, torch.tensor(np.asarray(offs, np.int32), **i32), torch.tensor(np.asarray(nq, np.int32), **i32),
                      torch.tensor(np.asarray(toks, np.int32), **i32), max(nq),
                      torch.tensor(np.asarray(ctx, np.int32), **i32), tau,
                      torch.from_numpy(np.asarray(u, np.float32)).cuda(), seed, *out, ws, st)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out] + [int(st.item())]


@pytest.mark.parametrize("vocab", [1000, 50_257, qi.VOCAB])
@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("tau", [0.6, 1.0])
def test_sample_accept_matches_oracle(vocab, bf16, tau):
    rng = np.random.default_rng(vocab + int(10 * tau) + 3 * bf16)
    nq = [int(x) for x in rng.integers(0, 17, size=8)]
    nq[1], nq[5] = 0, 1
    offs = np.concatenate([[0], np.cumsum(nq)[:-1]]).astype(np.int32)
    rows = int(sum(nq))
    logits = qi.logits_rows(vocab + 1, rows, vocab, "normal", bf16)
    lg64 = logits.astype(np.float64)
    # drafts drawn from each row's top tokens, so acceptance probabilities are sizeable
    toks = qi.random_tokens(vocab, rows, vocab)
    top = np.argsort(-lg64, axis=1)[:, :3]
    for b, T in enumerate(nq):
        for j in range(1, T):
            toks[offs[b] + j] = top[offs[b] + j - 1, int(rng.integers(0, 3))]
    # uniforms, kept clear of each draft test's boundary
    u = rng.uniform(0.0, 1.0, size=rows)
    for b, T in enumerate(nq):
        for j in range(T - 1):
            r = offs[b] + j
            p = target_prob(lg64[r], tau, int(toks[r + 1]))
            while abs(u[r] - p) < 2e-3:
                u[r] = rng.uniform()
    u = u.astype(np.float32)
    ctx = [int(x) for x in rng.integers(20, 5000, size=8)]
    seed = 0x1234_5678_9ABC_DEF0 + vocab
    want = sample_accept(lg64, offs, nq, toks, ctx, tau, u.astype(np.float64), seed)
    n_acc, nxt, com, st = _run_sample(logits, offs, nq, toks, ctx, bf16, tau, u, seed)
    assert st == 0
    assert np.array_equal(n_acc, want[0]) and np.array_equal(com, want[2])
    for b, T in enumerate(nq):
        if T == 0:
            assert nxt[b] == -1
            continue
        if nxt[b] == want[1][b]:
            continue
        # a different token must still be a maximal Gumbel key up to rounding
        r = offs[b] + int(n_acc[b])
        keys = gumbel_keys(lg64[r], tau, seed, r)
        if n_acc[b] < T - 1:
            keys[int(toks[r + 1])] = -np.inf
        assert keys[nxt[b]] >= keys.max() - 1e-4, (b, nxt[b], want[1][b])


def test_sample_accept_low_temperature_is_greedy():
    vocab = 4099
    nq = [6, 3, 1]
    offs = [0, 6, 9]
    logits = qi.logits_rows(11, 10, vocab)
    toks = _plant(logits, offs, nq, [3, 2, 0], 11, vocab)
    ctx = [100, 50, 7]
    u = np.random.default_rng(2).uniform(0.01, 0.99, size=10).astype(np.float32)
    want = greedy_accept(logits.astype(np.float64), offs, nq, toks, ctx)
    n_acc, nxt, com, st = _run_sample(logits, offs, nq, toks, ctx, False, 1e-3, u, 5)
    assert st == 0
    assert np.array_equal(n_acc, want[0]) and np.array_equal(nxt, want[1]) and np.array_equal(com, want[2])


# ----------------------------------------------------------------------------- top-p nucleus
from oracle.accept import nucleus_cut, sample_accept_nucleus


def _run_nucleus(logits_np, offs, nq, toks, ctx, bf16, tau, top_p, u, seed):
    from speculative_verify_attention_q3kv_gb300 import api
    rows, vocab = logits_np.shape
    lg = torch.from_numpy(logits_np).cuda()
    if bf16:
        lg = lg.to(torch.bfloat16)
    i32 = dict(dtype=torch.int32, device="cuda")
    S = len(nq)
    out = [torch.full((S,), -7, **i32) for _ in range(3)]
    ws = torch.empty(max(api.accept_workspace_bytes(rows, vocab), 8), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, **i32)
    api.accept_sample_nucleus(lg, torch.tensor(np.asarray(offs, np.int32), **i32),
                              torch.tensor(np.asarray(nq, np.int32), **i32), torch.tensor(np.asarray(toks, np.int32), **i32),
                              max(nq), torch.tensor(np.asarray(ctx, np.int32), **i32), tau, top_p,
                              torch.from_numpy(np.asarray(u, np.float32)).cuda(), seed, *out, ws, st)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out] + [int(st.item())]


def _clear_of_cut(lg64, tau, top_p, margin=1e-5):
    """top_p is not within `margin` of a row's cumulative mass at its cut or just above it."""
    for row in lg64:
        p = np.exp(row / tau - np.max(row / tau))
        p /= p.sum()
        cut, mass = nucleus_cut(row, tau, top_p)
        above = float(p[row > cut].sum())
        if abs(mass - top_p) < margin or abs(top_p - above) < margin:
            return False
    return True


@pytest.mark.parametrize("vocab", [1000, 50_257, qi.VOCAB])
@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("top_p", [0.5, 0.9])
def test_nucleus_accept_matches_oracle(vocab, bf16, top_p):
    tau = 0.8
    rng = np.random.default_rng(vocab + int(100 * top_p) + 7 * bf16)
    nq = [int(x) for x in rng.integers(0, 17, size=8)]
    nq[1], nq[5] = 0, 1
    offs = np.concatenate([[0], np.cumsum(nq)[:-1]]).astype(np.int32)
    rows = int(sum(nq))
    # sharp rows (scale 4) so the nuclei are a few hundred tokens at most
    logits = (qi.logits_rows(vocab + 5, rows, vocab, "normal", False) * 4.0).astype(np.float32)
    if bf16:
        logits = torch.from_numpy(logits).to(torch.bfloat16).float().numpy()
    lg64 = logits.astype(np.float64)
    while not _clear_of_cut(lg64, tau, top_p):
        top_p = float(top_p + 1e-4)
    toks = qi.random_tokens(vocab, rows, vocab)
    top = np.argsort(-lg64, axis=1)[:, :4]
    for b, T in enumerate(nq):
        for j in range(1, T):
            toks[offs[b] + j] = top[offs[b] + j - 1, int(rng.integers(0, 4))]
    u = rng.uniform(0.0, 1.0, size=rows)
    for b, T in enumerate(nq):
        for j in range(T - 1):
            r = offs[b] + j
            cut, mass = nucleus_cut(lg64[r], tau, top_p)
            d = int(toks[r + 1])
            q = target_prob(lg64[r], tau, d) / mass if lg64[r, d] >= cut else 0.0
            while abs(u[r] - q) < 2e-3:
                u[r] = rng.uniform()
    u = u.astype(np.float32)
    ctx = [int(x) for x in rng.integers(20, 5000, size=8)]
    seed = 0x0F0F_1234_5678_9ABC + vocab
    want = sample_accept_nucleus(lg64, offs, nq, toks, ctx, tau, top_p, u.astype(np.float64), seed)
    n_acc, nxt, com, st = _run_nucleus(logits, offs, nq, toks, ctx, bf16, tau, top_p, u, seed)
    assert st == 0
    assert np.array_equal(n_acc, want[0]) and np.array_equal(com, want[2])
    for b, T in enumerate(nq):
        if T == 0:
            assert nxt[b] == -1
            continue
        r = offs[b] + int(n_acc[b])
        cut, _ = nucleus_cut(lg64[r], tau, top_p)
        assert lg64[r, nxt[b]] >= cut                   # always inside the nucleus
        if nxt[b] == want[1][b]:
            continue
        keys = gumbel_keys(lg64[r], tau, seed, r)
        keys[lg64[r] < cut] = -np.inf
        if n_acc[b] < T - 1:
            keys[int(toks[r + 1])] = -np.inf
        assert keys[nxt[b]] >= keys.max() - 1e-4, (b, nxt[b], want[1][b])


def test_nucleus_top_p_one_and_ties():
    vocab = 3001
    nq = [5, 4]
    offs = [0, 5]
    rows = 9
    # values on a 0.5 grid: many exact ties, also at the cut
    logits = (np.round(qi.logits_rows(17, rows, vocab, "normal", False) * 6) / 2).astype(np.float32)
    lg64 = logits.astype(np.float64)
    toks = qi.random_tokens(3, rows, vocab)
    u = np.full(rows, 0.5, np.float32)
    ctx = [40, 41]
    # top_p = 1: the plain sampled acceptance
    a1 = _run_nucleus(logits, offs, nq, toks, ctx, False, 1.0, 1.0, u, 9)
    a0 = _run_sample(logits, offs, nq, toks, ctx, False, 1.0, u, 9)
    for x, y in zip(a1, a0):
        assert np.array_equal(x, y)
    # ties at the cut are kept: the chosen token is in the oracle's (threshold) nucleus
    for top_p in (0.05, 0.3):
        while not _clear_of_cut(lg64, 1.0, top_p):
            top_p += 1e-4
        uu = u.copy()
        for b, T in enumerate(nq):
            for j in range(T - 1):
                r = offs[b] + j
                cut, mass = nucleus_cut(lg64[r], 1.0, top_p)
                d = int(toks[r + 1])
                q = target_prob(lg64[r], 1.0, d) / mass if lg64[r, d] >= cut else 0.0
                if abs(uu[r] - q) < 2e-3:
                    uu[r] = 0.9 if q < 0.5 else 0.1
        n_acc, nxt, com, st = _run_nucleus(logits, offs, nq, toks, ctx, False, 1.0, top_p, uu, 9)
        want = sample_accept_nucleus(lg64, offs, nq, toks, ctx, 1.0, top_p, uu.astype(np.float64), 9)
        assert st == 0 and np.array_equal(n_acc, want[0]) and np.array_equal(com, want[2])
        for b, T in enumerate(nq):
            r = offs[b] + int(n_acc[b])
            cut, _ = nucleus_cut(lg64[r], 1.0, top_p)
            assert lg64[r, nxt[b]] >= cut
            if nxt[b] != want[1][b]:
                keys = gumbel_keys(lg64[r], 1.0, 9, r)
                keys[lg64[r] < cut] = -np.inf
                if n_acc[b] < T - 1:
                    keys[int(toks[r + 1])] = -np.inf
                assert keys[nxt[b]] >= keys.max() - 1e-4
