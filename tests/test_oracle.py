"""Pins of the fp64 oracle against what the FlashPrefill V2 paper and mathematics fix.

Nothing here compares the oracle with itself: each test checks it against a
library routine (torch softmax attention, torch's bf16 / float8_e4m3fn
conversions), a closed form, an invariant or a second brute-force
implementation written in a different algebraic form, so that a plausible
slip in the oracle (a dropped 1/sqrt(d), a sum for a mean, log2 for ln, an
off-by-one window, ">" for ">=", a wrong correction set) fails at least one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_sparse_long_mean_gb300 import synth

D = 128


# ----------------------------------------------------------------- helpers

def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def paged_problem(q, ks, vs, hq, hkv, page=64, seed=0, permute=True, dtype="bf16", scales=(1.0, 1.0, 1.0),
                  tile_rows=128):
    """Problem from contiguous per-request keys/values ([L_b, hkv, d] raw element arrays)."""
    lengths = [k.shape[0] for k in ks]
    npg = [(L + page - 1) // page for L in lengths]
    total = sum(npg) + 3
    rng = np.random.default_rng(seed)
    perm = rng.permutation(total) if permute else np.arange(total)
    pt = np.full((len(lengths), max(max(npg), 1)), -1, np.int32)
    elem = ks[0].dtype
    kp = np.zeros((total, page, hkv, D), dtype=elem)
    vp = np.zeros((total, page, hkv, D), dtype=elem)
    off = 0
    for b, L in enumerate(lengths):
        pt[b, :npg[b]] = perm[off:off + npg[b]]
        off += npg[b]
        for j in range(L):
            kp[pt[b, j // page], j % page] = ks[b][j]
            vp[pt[b, j // page], j % page] = vs[b][j]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return oracle.Problem(q=q, k_pages=kp, v_pages=vp, cu_seqlens=cu, page_table=pt, hq=hq, hkv=hkv, dtype=dtype,
                          c_q=scales[0], c_k=scales[1], c_v=scales[2], tile_rows=tile_rows)


def dequant(p: oracle.Problem, raw, scale):
    if p.dtype == "bf16":
        return torch.from_numpy(raw.view(np.int16).copy()).view(torch.bfloat16).double()
    return torch.from_numpy(raw.copy()).view(torch.float8_e4m3fn).double() * scale


def gathered(p: oracle.Problem, b: int):
    """Contiguous fp64 K, V [L^kv, hkv, d] of request b, gathered by plain indexing."""
    L = int(p.kv_lengths()[b])
    j = np.arange(L)
    pages = p.page_table[b, j // p.page_size]
    K = dequant(p, p.k_pages[pages, j % p.page_size], p.c_k)
    V = dequant(p, p.v_pages[pages, j % p.page_size], p.c_v)
    return K, V


def torch_dense_causal(p: oracle.Problem):
    """Textbook causal softmax attention, per request and query head, via torch; the L^q queries are the
    last positions of the L^kv keys (bottom-right aligned causal mask)."""
    Q = dequant(p, p.q, p.c_q)
    out = torch.zeros_like(Q)
    for b in range(p.batch):
        s, e = int(p.cu_seqlens[b]), int(p.cu_seqlens[b + 1])
        if e == s:
            continue
        K, V = gathered(p, b)
        Lkv = K.shape[0]
        for hh in range(p.hq):
            kv = hh // p.g
            logits = Q[s:e, hh] @ K[:, kv].T / math.sqrt(D)
            mask = torch.ones(e - s, Lkv, dtype=torch.bool).tril(diagonal=Lkv - (e - s))
            logits = logits.masked_fill(~mask, float("-inf"))
            out[s:e, hh] = torch.softmax(logits, dim=-1) @ V[:, kv]
    return out.numpy()


def rel_err(a, b):
    a, b = np.asarray(a, float), np.asarray(b, float)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def small_workload(lengths=(300, 200), hq=8, hkv=2, mu_scale=0.5, seed=1, paging="random", dtype="bf16",
                   stripes=False, kv_lengths=None):
    return synth.make_workload("tiny_2k", lengths=list(lengths), hq=hq, hkv=hkv, mu_scale=mu_scale, seed=seed,
                               paging=paging, dtype=dtype, stripes=stripes,
                               kv_lengths=None if kv_lengths is None else list(kv_lengths))


# ------------------------------------------------------ element decoding

def test_bf16_decode_matches_torch_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    L = oracle.lib()
    got = np.array([L.orc_decode_bf16(int(x)) for x in bits[::97]] + [L.orc_decode_bf16(int(x)) for x in
                                                                     range(0x3F00, 0x4100)])
    want = np.concatenate([ref[::97], ref[0x3F00:0x4100]])
    both_nan = np.isnan(got) & np.isnan(want)
    assert np.all(both_nan | (got == want))


def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.lib().orc_decode_e4m3(int(c)) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.nanmax(got) == 448.0 and np.nanmin(got) == -448.0


# ----------------------------------------------------------- pooling (Eq.5)

def test_pool_closed_form_with_ragged_last_block_and_permuted_pages():
    # keys: token j of the block has every coordinate equal to (j mod 128) + 1 (exact in bf16);
    # values: coordinate c of token j equals c - 64. Means follow in closed form.
    L = 128 * 2 + 37
    j = np.arange(L)
    k = np.repeat(((j % 128) + 1.0)[:, None], D, axis=1)[:, None, :]
    v = np.tile((np.arange(D) - 64.0)[None, :], (L, 1))[:, None, :]
    q = bf16_bits(torch.zeros(L, 1, D))
    p = paged_problem(q, [bf16_bits(torch.from_numpy(k))], [bf16_bits(torch.from_numpy(v))], hq=1, hkv=1, seed=3)
    pooled = oracle.pool(p)
    assert list(pooled.cnt) == [128, 128, 37]
    np.testing.assert_array_equal(pooled.kbar[:, 0, 0], [64.5, 64.5, 19.0])   # mean of 1..n
    np.testing.assert_array_equal(pooled.vbar[:, 0], np.tile(np.arange(D) - 64.0, (3, 1)))


def test_am_gm_lower_bound_of_pooled_score():
    # exp(q.kbar/sqrt d) <= (1/|B_J|) sum_i exp(q.k_i/sqrt d)   (Sec.3.1; FlashPrefill Sec.3.1)
    w = small_workload(lengths=(384,), hq=4, hkv=1, mu_scale=1.0)
    p = oracle.Problem.from_workload(w)
    pooled = oracle.pool(p)
    K, _ = gathered(p, 0)
    Q = dequant(p, p.q, 1.0)[:, 0]
    nb = 3
    for J in range(nb):
        kb = torch.from_numpy(pooled.kbar[J, 0])
        pooled_score = torch.exp(Q @ kb / math.sqrt(D))
        exact = torch.exp(Q @ K[J * 128:(J + 1) * 128, 0].T / math.sqrt(D)).mean(dim=1)
        assert torch.all(pooled_score <= exact * (1 + 1e-12))
        # and the bound is not trivially loose: a summed (not averaged) key would break it
        assert torch.any(torch.exp(Q @ (kb * 128) / math.sqrt(D)) > exact)


# --------------------------------------------------- selection (Eq.3, Eq.20)

def _select(E, D_, alpha, sink, window):
    E = np.asarray(E, dtype=np.float64)
    sel = np.zeros(D_ + 1, np.uint8)
    near = np.zeros(D_ + 1, np.uint8)
    n = oracle.lib().orc_select(oracle._ptr(E), D_, alpha, sink, window, oracle._ptr(sel), oracle._ptr(near))
    return n, sel, near


def test_threshold_is_inclusive_and_near_flags():
    # D = 6; block 6 is the diagonal; with sink=1 and window=1 blocks 0, 5, 6 are forced.
    E = [0.0, 0.1, 0.09995, 0.0999, 0.2, 0.0, 1.0]
    n, sel, near = _select(E, 6, 0.1, 1, 1)
    assert list(sel) == [1, 1, 0, 0, 1, 1, 1]          # E >= 0.1 * 1.0 kept, ties included
    assert list(near) == [0, 1, 1, 0, 0, 0, 0]          # |E - thr| <= 1e-3 thr, forced blocks excluded
    assert n == 5


def test_forced_blocks_and_alpha_limits():
    D_ = 9
    E = np.array([3.0, 1.0, 8.0, 0.5, 0.25, 9.0, 0.1, 0.3, 0.2, 0.05])
    # alpha > 1 keeps only the forced set
    _, sel, _ = _select(E, D_, 1.5, 2, 3)
    assert list(np.nonzero(sel)[0]) == [0, 1, 6, 7, 8, 9]
    # alpha = 1 keeps the argmax (block 5) and the forced set
    _, sel, _ = _select(E, D_, 1.0, 0, 0)
    assert list(np.nonzero(sel)[0]) == [5, 9]
    # alpha = 0 keeps everything causal
    _, sel, _ = _select(E, D_, 0.0, 0, 0)
    assert sel.all()
    # window larger than D clips at block 0
    _, sel, _ = _select(E[:3], 2, 2.0, 0, 10)
    assert sel.all()


def test_selection_monotone_in_alpha():
    w = small_workload(lengths=(512, 256), hq=8, hkv=2, mu_scale=0.5)
    p = oracle.Problem.from_workload(w)
    seg = oracle.segments(p)
    pooled = oracle.pool(p, seg)
    prev = None
    for a in [0.0, 0.01, 0.05, 0.2, 0.5, 1.0]:
        s = oracle.select(p, a, 1, 1, seg=seg, pooled=pooled).sel_full
        if prev is not None:
            assert np.all(s <= prev)
        prev = s


# ------------------------------------------------------- P1: alpha = 0 = dense

@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_alpha_zero_reproduces_dense_causal_attention(dtype):
    w = small_workload(lengths=(300, 200, 77), hq=8, hkv=2, mu_scale=0.5, dtype=dtype)
    p = oracle.Problem.from_workload(w)
    ref = torch_dense_causal(p)
    res = oracle.run(p, alpha=0.0, sink=1, window=1)
    assert rel_err(res["O"], ref) < 1e-12
    # every causal block is selected: CSR = all J <= D
    seg = res["seg"]
    assert len(res["idx"]) == int((seg.D + 1).sum())
    # the dense flag gives the same output whatever the selection
    res2 = oracle.run(p, alpha=0.9, sink=0, window=0, dense=True)
    assert rel_err(res2["O"], ref) < 1e-12


def test_lse_matches_torch_logsumexp_in_dense_mode():
    w = small_workload(lengths=(256,), hq=4, hkv=1)
    p = oracle.Problem.from_workload(w)
    res = oracle.run(p, alpha=0.0, sink=0, window=0)
    Q = dequant(p, p.q, 1.0)
    K, _ = gathered(p, 0)
    for hh in range(4):
        logits = Q[:, hh] @ K[:, 0].T / math.sqrt(D)
        logits = logits.masked_fill(~torch.ones(256, 256, dtype=torch.bool).tril(), float("-inf"))
        np.testing.assert_allclose(res["lse"][:, hh], torch.logsumexp(logits, -1).numpy(), rtol=1e-13, atol=1e-12)


# ------------------------------------- P2: identical blocks make the surrogate exact

def test_identical_blocks_make_mean_correction_exact():
    # Every token of block J carries the same key and value, so |B_J| e^{q.kbar/sqrt d} vbar equals
    # the block's exact contribution (Sec.3.2 Eq.7 with delta = 0): the corrected output equals dense
    # attention for any alpha, while the uncorrected one (Eq.4) does not.
    torch.manual_seed(5)
    hq, hkv, g = 4, 1, 4
    lengths = [640, 384]
    ks, vs, qs = [], [], []
    for L in lengths:
        nb = (L + 127) // 128
        kc = torch.randn(nb, hkv, D)
        vc = torch.randn(nb, hkv, D)
        blk = torch.arange(L) // 128
        ks.append(bf16_bits(kc[blk]))
        vs.append(bf16_bits(vc[blk]))
        # queries lean towards their own block's key, so off-diagonal blocks fall below the threshold
        qs.append(1.5 * kc[blk, 0][:, None, :] + 0.5 * torch.randn(L, hq, D))
    q = bf16_bits(torch.cat(qs))
    p = paged_problem(q, ks, vs, hq=hq, hkv=hkv, seed=9)
    ref = torch_dense_causal(p)
    for alpha in [0.3, 1.0, 2.0]:
        res = oracle.run(p, alpha=alpha, sink=0, window=0, correction=True)
        assert rel_err(res["O"], ref) < 1e-12, alpha
        assert len(res["idx"]) < int((res["seg"].D + 1).sum())    # something really was pruned
        nocorr = oracle.run(p, alpha=alpha, sink=0, window=0, correction=False)
        assert rel_err(nocorr["O"], ref) > 1e-6, alpha


def test_two_block_closed_form():
    # L = 256, g = 1: tile 1 (positions 128..255) has D = 1. Block 0 keys are a*e0, block 1 keys b*e0,
    # queries c*e0, block values v0 / v1. With sink = window = 0 block 0 is pruned iff
    # exp(c (a - b) / sqrt d) < alpha, and then its surrogate weight is 128 e^{c a / sqrt d}.
    a, bk, c = 1.0, 3.0, 2.0
    L = 256
    e0 = torch.zeros(D)
    e0[0] = 1.0
    k = torch.cat([a * e0.expand(128, D), bk * e0.expand(128, D)])[:, None]
    v0, v1 = torch.full((D,), 0.5), torch.full((D,), -1.25)
    v = torch.cat([v0.expand(128, D), v1.expand(128, D)])[:, None]
    q = (c * e0).expand(L, 1, D)
    p = paged_problem(bf16_bits(q), [bf16_bits(k)], [bf16_bits(v)], hq=1, hkv=1, seed=2)
    ratio = math.exp(c * (a - bk) / math.sqrt(D))           # E_0 / E_1 for tile 1
    sa, sb = c * a / math.sqrt(D), c * bk / math.sqrt(D)
    for alpha, pruned in [(ratio * 0.999, False), (ratio * 1.001, True)]:
        for corr in (True, False):
            res = oracle.run(p, alpha=alpha, sink=0, window=0, correction=corr)
            sel1 = res["selection"].selected(res["seg"], 1)
            assert list(sel1) == ([1] if pruned else [0, 1])
            for pos in (128, 200, 255):
                n1 = pos - 127
                w0 = 128 * math.exp(sa) if (not pruned or corr) else 0.0
                w1 = n1 * math.exp(sb)
                want = (w0 * 0.5 + w1 * -1.25) / (w0 + w1)
                np.testing.assert_allclose(res["O"][pos, 0], want, rtol=1e-13)
                np.testing.assert_allclose(res["lse"][pos, 0], math.log(w0 + w1), rtol=1e-13)


# ---------------------------------- P4: brute force in the Eq.1-2 form, L <= 512

def brute_force(p: oracle.Problem, alpha, sink, window, correction=True):
    """Materialises the whole [rows x blocks] pooled-logit matrix per (request, KV head) and
    selects with the per-(tile, block) maxima m_IJ, M_I and the normalised Score of Eq.1-2 (eps = 0);
    attention enumerates each row's token set explicitly. Query rows are keyed by absolute position
    (the new tokens are the last L^q of L^kv) and grouped into tiles by the absolute packed row
    g pos + head mod g; the result is keyed by (request, KV head, absolute tile)."""
    Q = dequant(p, p.q, p.c_q)
    out = np.zeros(Q.shape)
    sels = {}
    Lq_all, Lkv_all = p.lengths(), p.kv_lengths()
    for b in range(p.batch):
        s0, Lq, L = int(p.cu_seqlens[b]), int(Lq_all[b]), int(Lkv_all[b])
        if Lq == 0:
            continue
        shift = L - Lq
        K, V = gathered(p, b)
        nb = (L + 127) // 128
        cnt = torch.tensor([min(128, L - 128 * J) for J in range(nb)], dtype=torch.float64)
        kbar = torch.stack([K[128 * J:128 * J + int(cnt[J])].mean(0) for J in range(nb)])   # [nb, hkv, d]
        vbar = torch.stack([V[128 * J:128 * J + int(cnt[J])].mean(0) for J in range(nb)])
        for h in range(p.hkv):
            pos = torch.arange(shift, L).repeat_interleave(p.g)       # absolute position of each query row
            head = h * p.g + torch.arange(p.g).repeat(Lq)
            tok = s0 + pos - shift                                    # row of q holding that query
            Qp = Q[tok, head]                                         # packed Q' rows [g L^q, d]
            logits = Qp @ kbar[:, h].T / math.sqrt(D)                 # [g L^q, nb]
            tile = (p.g * pos + head % p.g) // 128
            for T in torch.unique(tile).tolist():
                r = torch.nonzero(tile == T).flatten()
                Dg = int(pos[r[0]]) // 128
                assert int(pos[r[-1]]) // 128 == Dg
                lg = logits[r, :Dg + 1]
                m_IJ = lg.max(0).values
                S_IJ = torch.exp(lg - m_IJ).sum(0)
                M_I = m_IJ.max()
                score = S_IJ * torch.exp(m_IJ - M_I)
                score = score / score.sum()
                thresh = alpha * score.max()
                J = torch.arange(Dg + 1)
                forced = (J < sink) | ((J >= Dg - window) & (J < Dg)) | (J == Dg)
                sel = (score >= thresh) | forced
                sels[(b, h, T)] = sel.numpy()
                for rr in r.tolist():
                    ps, hh, tr = int(pos[rr]), int(head[rr]), int(tok[rr])
                    toks = [j for Jb in range(Dg + 1) if sel[Jb] for j in range(128 * Jb, min(128 * Jb + 128, L))
                            if j <= ps]
                    toks = torch.tensor(toks)
                    lt = Q[tr, hh] @ K[toks, h].T / math.sqrt(D)
                    vals = V[toks, h]
                    if correction:
                        C = [Jb for Jb in range(Dg) if not sel[Jb]]
                        if C:
                            C = torch.tensor(C)
                            lt = torch.cat([lt, Q[tr, hh] @ kbar[C, h].T / math.sqrt(D) + torch.log(cnt[C])])
                            vals = torch.cat([vals, vbar[C, h]])
                    out[tr, hh] = (torch.softmax(lt, 0) @ vals).numpy()
    return sels, out


@pytest.mark.parametrize("hq,hkv,lengths,alpha,sink,window", [
    (4, 1, (512,), 0.1, 1, 1),
    (8, 2, (300, 211), 0.05, 0, 0),
    (8, 1, (512, 129), 0.3, 1, 0),
    (2, 2, (512,), 0.02, 1, 0),
])
def test_brute_force_agrees(hq, hkv, lengths, alpha, sink, window):
    w = small_workload(lengths=lengths, hq=hq, hkv=hkv, mu_scale=0.6, seed=hq * 7 + len(lengths))
    p = oracle.Problem.from_workload(w)
    res = oracle.run(p, alpha=alpha, sink=sink, window=window)
    sels, ref = brute_force(p, alpha, sink, window)
    seg = res["seg"]
    nonforced_pruned = 0
    for s in range(len(seg)):
        key = (int(seg.b[s]), int(seg.h[s]), int(seg.T[s]))
        o = seg.full_off[s]
        mine = res["selection"].sel_full[o:o + seg.D[s] + 1]
        near = res["selection"].near_full[o:o + seg.D[s] + 1]
        diff = (mine != sels[key].astype(np.uint8))
        assert not np.any(diff & (near == 0)), key
        nonforced_pruned += int((mine == 0).sum())
    assert nonforced_pruned > 0
    assert rel_err(res["O"], ref) < 1e-12


def test_uncorrected_matches_brute_force():
    w = small_workload(lengths=(512,), hq=4, hkv=1, mu_scale=0.4, seed=3)
    p = oracle.Problem.from_workload(w)
    res = oracle.run(p, alpha=0.1, sink=1, window=1, correction=False)
    _, ref = brute_force(p, 0.1, 1, 1, correction=False)
    assert rel_err(res["O"], ref) < 1e-12


# ------------------------------------------------ P6: paging and batching invariance

def test_page_permutation_and_request_order_invariance():
    w = small_workload(lengths=(300, 200, 129), hq=8, hkv=2, mu_scale=0.5, seed=4)
    p = oracle.Problem.from_workload(w)
    base = oracle.run(p, alpha=0.1, sink=1, window=1)
    # 1) move every page to a new slot
    rng = np.random.default_rng(0)
    n = p.k_pages.shape[0]
    perm = rng.permutation(n)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(n)
    kp = p.k_pages[perm]
    vp = p.v_pages[perm]
    pt = np.where(p.page_table >= 0, inv[np.maximum(p.page_table, 0)], -1).astype(np.int32)
    p2 = oracle.Problem(q=p.q, k_pages=kp, v_pages=vp, cu_seqlens=p.cu_seqlens, page_table=pt, hq=p.hq, hkv=p.hkv)
    r2 = oracle.run(p2, alpha=0.1, sink=1, window=1)
    assert np.array_equal(base["cu"], r2["cu"]) and np.array_equal(base["idx"], r2["idx"])
    assert np.array_equal(base["O"], r2["O"])
    # 2) reverse the request order
    order = [2, 1, 0]
    L = p.lengths()
    qs = [p.q[p.cu_seqlens[b]:p.cu_seqlens[b + 1]] for b in order]
    cu = np.concatenate([[0], np.cumsum(L[order])]).astype(np.int32)
    p3 = oracle.Problem(q=np.concatenate(qs), k_pages=p.k_pages, v_pages=p.v_pages, cu_seqlens=cu,
                        page_table=p.page_table[order], hq=p.hq, hkv=p.hkv)
    r3 = oracle.run(p3, alpha=0.1, sink=1, window=1)
    for new_b, old_b in enumerate(order):
        a0, a1 = p.cu_seqlens[old_b], p.cu_seqlens[old_b + 1]
        n0 = cu[new_b]
        assert np.array_equal(base["O"][a0:a1], r3["O"][n0:n0 + (a1 - a0)])


# ------------------------------------------------------------ P7: closed forms

def test_csr_index_memory_matches_paper_table7_under_packed_tiles():
    # Tab.7: at batch 1, 32 query heads, 4 KV heads, a CSR of 64-token int32 tiles takes about
    # 3 MB at 64K (9% density) and 6 MB at 128K (5%). The segment structure of the oracle (tiles of
    # 128 packed rows per KV head) reproduces those sizes; tiles of 128 positions would not.
    for L, rho, mb in [(65536, 0.09, 3.0), (131072, 0.05, 6.0)]:
        p = oracle.Problem(q=np.zeros((1, 32, D), np.uint16), k_pages=np.zeros((1, 64, 4, D), np.uint16),
                           v_pages=np.zeros((1, 64, 4, D), np.uint16), cu_seqlens=np.array([0, L], np.int32),
                           page_table=np.zeros((1, 1), np.int32), hq=32, hkv=4)
        seg = oracle.segments(p)
        assert len(seg) == 4 * (8 * L // 128)
        causal_pairs = int((seg.D + 1).sum())
        bytes_ = rho * causal_pairs * 2 * 4
        assert abs(bytes_ / 2 ** 20 - mb) / mb < 0.1, (L, bytes_)
        dense_mask = 32 * (L // 128) ** 2
        assert dense_mask == {65536: 8, 131072: 32}[L] * 2 ** 20


def test_overhead_ratio_closed_form():
    # Eq.24: (C_idx + C_corr) / C_attn = (2 - rho) / (2 rho B) ~ 19% at rho = 4%, B = 128.
    rho, B = 0.04, 128
    assert abs((2 - rho) / (2 * rho * B) - 0.1914) < 1e-3


# ----------------------------------------------- approximation quality (soft)

def test_correction_reduces_error_on_the_generator():
    w = small_workload(lengths=(1024,), hq=4, hkv=1, mu_scale=1.0, seed=8, paging="identity")
    p = oracle.Problem.from_workload(w)
    dense = oracle.run(p, alpha=0.0, sink=1, window=1)["O"]
    corr = oracle.run(p, alpha=0.1, sink=1, window=1, correction=True)["O"]
    nocorr = oracle.run(p, alpha=0.1, sink=1, window=1, correction=False)["O"]
    assert np.linalg.norm(corr - dense) < np.linalg.norm(nocorr - dense)


# ------------------------------------------- 64-token tile CSR (serving format)

def test_tiles64_hand_example_and_token_enumeration():
    """Block J of a request covers the 64-token tiles holding any of its tokens (Sec.3.4, Alg.1 step 5)."""
    w = small_workload(lengths=(300, 64, 129), hq=4, hkv=1)
    op = oracle.Problem.from_workload(w)
    seg = oracle.segments(op)
    # request 0: L = 300 -> blocks 0..2 cover tiles {0, 1}, {2, 3}, {4} (tokens 256..299 lie in tile 4 only)
    s0 = int(np.nonzero(seg.b == 0)[0][-1])   # the last tile of request 0 reaches block 2
    assert seg.D[s0] == 2
    cu = np.zeros(len(seg) + 1, np.int32)
    parts = []
    rng = np.random.default_rng(7)
    for s in range(len(seg)):
        ids = np.array([0, 1, 2], np.int32) if s == s0 else np.sort(
            rng.choice(seg.D[s] + 1, size=rng.integers(1, seg.D[s] + 2), replace=False)).astype(np.int32)
        parts.append(ids)
        cu[s + 1] = cu[s] + len(ids)
    idx = np.concatenate(parts)
    tcu, tidx = oracle.tiles64_from_csr(op, seg, cu, idx)
    assert list(tidx[tcu[s0]:tcu[s0 + 1]]) == [0, 1, 2, 3, 4]
    L = op.lengths()
    for s in range(len(seg)):
        # explicit token enumeration: every token of every selected block, mapped to its tile
        toks = np.concatenate([np.arange(128 * J, min(128 * J + 128, L[seg.b[s]])) for J in idx[cu[s]:cu[s + 1]]])
        want = np.unique(toks // 64)
        assert np.array_equal(tidx[tcu[s]:tcu[s + 1]], want), s
        # closed form of the count: two tiles per block, one for a block with at most 64 tokens
        n = sum(2 if 128 * J + 64 < L[seg.b[s]] else 1 for J in idx[cu[s]:cu[s + 1]])
        assert tcu[s + 1] - tcu[s] == n


# ------------------------------ P8: chunked prefill after a cached prefix (L^q < L^kv)

PREFIX_CASES = [
    # (L^q, L^kv) per request; g = 4 puts 32 positions in a tile
    ((200, 77, 1, 0, 130), (456, 300, 129, 64, 130)),   # prefix on / off the tile grid, one query, empty chunk
    ((300,), (1000,)),                                   # several prefix blocks, ragged KV tail
]


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("case", range(len(PREFIX_CASES)))
def test_prefix_dense_matches_textbook_causal_attention(dtype, case):
    # With alpha = 0 every causal block is exact, so each new query at absolute position L^kv - L^q + i
    # must see exactly keys 0 .. L^kv - L^q + i of the whole KV (bottom-right aligned causal mask).
    lq, lkv = PREFIX_CASES[case]
    w = small_workload(lengths=lq, kv_lengths=lkv, hq=8, hkv=2, mu_scale=0.5, dtype=dtype, seed=11 + case)
    p = oracle.Problem.from_workload(w)
    ref = torch_dense_causal(p)
    res = oracle.run(p, alpha=0.0, sink=1, window=1)
    assert rel_err(res["O"], ref) < 1e-12
    assert not np.isnan(res["O"]).any()
    seg = res["seg"]
    assert len(res["idx"]) == int((seg.D + 1).sum())
    res2 = oracle.run(p, alpha=0.7, sink=0, window=0, dense=True)
    assert rel_err(res2["O"], ref) < 1e-12


def test_prefix_tile_geometry_hand_example():
    # g = 4, L^q = 77 after a 223-token prefix: query rows are absolute packed rows [4 * 223, 4 * 300)
    # = [892, 1200), i.e. tiles 6 .. 9 (tile 6 holds only position 223's 4 rows 892..895); tile T lies in
    # block floor(32 T / 128): blocks 1, 1, 2, 2. 300 keys pool into 3 blocks (128, 128, 44 tokens).
    w = small_workload(lengths=(77,), kv_lengths=(300,), hq=8, hkv=2, seed=4)
    p = oracle.Problem.from_workload(w)
    seg = oracle.segments(p)
    assert list(seg.T) == [6, 7, 8, 9] * 2 and list(seg.t) == [0, 1, 2, 3] * 2
    assert list(seg.D) == [1, 1, 2, 2] * 2
    assert seg.total_blocks == 3
    pooled = oracle.pool(p, seg)
    assert list(pooled.cnt[:3]) == [128, 128, 44]
    O, lse = oracle.attend(p, np.ones(seg.full_total, np.uint8), dense=True, seg=seg, seg_ids=[0, 3])
    # tile 6: only rows 892 - 768 = 124 .. 127 are query rows; tile 9 (rows 1152..1279): 48 rows
    assert [i for i in range(128) if lse[0, i] != 0] == [124, 125, 126, 127]
    assert int((lse[1] != 0).sum()) == 1200 - 1152


@pytest.mark.parametrize("hq,hkv,lq,lkv,alpha,sink,window", [
    (8, 2, (77, 200), (300, 456), 0.05, 1, 1),
    (4, 1, (260,), (777,), 0.1, 0, 0),
    (2, 2, (129, 1), (640, 513), 0.02, 1, 2),
])
def test_prefix_brute_force_agrees(hq, hkv, lq, lkv, alpha, sink, window):
    w = small_workload(lengths=lq, kv_lengths=lkv, hq=hq, hkv=hkv, mu_scale=0.6, seed=hq + sum(lq))
    p = oracle.Problem.from_workload(w)
    res = oracle.run(p, alpha=alpha, sink=sink, window=window)
    sels, ref = brute_force(p, alpha, sink, window)
    seg = res["seg"]
    assert len(sels) == len(seg)
    pruned = 0
    for s in range(len(seg)):
        key = (int(seg.b[s]), int(seg.h[s]), int(seg.T[s]))
        o = seg.full_off[s]
        mine = res["selection"].sel_full[o:o + seg.D[s] + 1]
        near = res["selection"].near_full[o:o + seg.D[s] + 1]
        assert not np.any((mine != sels[key].astype(np.uint8)) & (near == 0)), key
        pruned += int((mine == 0).sum())
    assert pruned > 0
    assert rel_err(res["O"], ref) < 1e-12


def test_chunked_prefill_reproduces_unchunked_tiles():
    # A chunk run sees the same queries as the unchunked prefill of the whole sequence and the same keys up
    # to the chunk's end, and its tiles sit on the same absolute grid: a tile of the chunk that holds only
    # chunk rows and whose diagonal block is complete within the chunk has the same pooled means, energies,
    # selection and output rows as that tile of the unchunked run. Every other row (the partial tile at the
    # chunk's start, tiles whose diagonal block the chunk cuts short) agrees in dense mode.
    full = small_workload(lengths=(700,), hq=8, hkv=2, mu_scale=0.6, seed=21)
    pf = oracle.Problem.from_workload(full)
    rf = oracle.run(pf, alpha=0.1, sink=1, window=1)
    df = oracle.run(pf, alpha=0.0, sink=0, window=0, dense=True)
    covered = np.zeros(700, bool)
    n_same = 0
    for lq_lo, lq_hi in [(0, 300), (300, 405), (405, 700)]:
        # the chunk: queries lq_lo .. lq_hi - 1 against the first lq_hi keys of the same paged KV
        pc = oracle.Problem(q=pf.q[lq_lo:lq_hi], k_pages=pf.k_pages, v_pages=pf.v_pages,
                            cu_seqlens=np.array([0, lq_hi - lq_lo], np.int32), page_table=pf.page_table,
                            hq=8, hkv=2, seqlens_kv=np.array([lq_hi], np.int32))
        rc = oracle.run(pc, alpha=0.1, sink=1, window=1)
        dc = oracle.run(pc, alpha=0.0, sink=0, window=0, dense=True)
        sf, sc = rf["seg"], rc["seg"]
        for s in range(len(sc)):
            T, h = int(sc.T[s]), int(sc.h[s])
            rows = np.arange(128 * T, 128 * T + 128)
            pos = rows // 4
            whole = pos.min() >= lq_lo
            fs = int(np.nonzero((sf.T == T) & (sf.h == h))[0][0])
            same = whole and pos.max() < lq_hi and 128 * (int(sc.D[s]) + 1) <= lq_hi
            if same:
                n_same += 1
                a = rc["selection"].sel_full[sc.full_off[s]:sc.full_off[s] + sc.D[s] + 1]
                b = rf["selection"].sel_full[sf.full_off[fs]:sf.full_off[fs] + sf.D[fs] + 1]
                np.testing.assert_array_equal(a, b)
            mine = (pos >= lq_lo) & (pos < lq_hi)
            heads = h * 4 + rows % 4
            for r in np.nonzero(mine)[0]:
                np.testing.assert_allclose(dc["O"][pos[r] - lq_lo, heads[r]], df["O"][pos[r], heads[r]],
                                           rtol=0, atol=1e-12)
                if same:
                    np.testing.assert_array_equal(rc["O"][pos[r] - lq_lo, heads[r]], rf["O"][pos[r], heads[r]])
                covered[pos[r]] = True
    assert covered.all() and n_same >= 20


def test_prefix_identical_blocks_make_mean_correction_exact():
    # Eq.7 with delta = 0 after a cached prefix: blocks of identical tokens make the corrected output equal
    # to dense causal attention over prefix + chunk for any alpha; the uncorrected one (Eq.4) differs.
    torch.manual_seed(6)
    hq, hkv = 4, 1
    lkv, lq = [900, 333], [250, 333]
    ks, vs, qs = [], [], []
    for L, n in zip(lkv, lq):
        nb = (L + 127) // 128
        kc, vc = torch.randn(nb, hkv, D), torch.randn(nb, hkv, D)
        blk = torch.arange(L) // 128
        ks.append(bf16_bits(kc[blk]))
        vs.append(bf16_bits(vc[blk]))
        qs.append((1.5 * kc[blk, 0][:, None, :] + 0.5 * torch.randn(L, hq, D))[L - n:])
    full = paged_problem(bf16_bits(torch.cat(qs)), ks, vs, hq=hq, hkv=hkv, seed=3)
    p = oracle.Problem(q=full.q, k_pages=full.k_pages, v_pages=full.v_pages,
                       cu_seqlens=np.concatenate([[0], np.cumsum(lq)]).astype(np.int32), page_table=full.page_table,
                       hq=hq, hkv=hkv, seqlens_kv=np.array(lkv, np.int32))
    ref = torch_dense_causal(p)
    for alpha in [0.3, 1.0]:
        res = oracle.run(p, alpha=alpha, sink=0, window=0, correction=True)
        assert rel_err(res["O"], ref) < 1e-12, alpha
        assert len(res["idx"]) < int((res["seg"].D + 1).sum())
        nocorr = oracle.run(p, alpha=alpha, sink=0, window=0, correction=False)
        assert rel_err(nocorr["O"], ref) > 1e-6, alpha


def test_prefix_validation_rejects_kv_shorter_than_queries():
    w = small_workload(lengths=(100,), hq=4, hkv=1)
    p = oracle.Problem.from_workload(w)
    p.seqlens_kv = np.array([99], np.int32)
    s = p.c_struct()
    import ctypes
    assert oracle.lib().orc_validate(ctypes.byref(s)) == -1


# -------------------------------------- P13: quantised FP8 probabilities (Eq.15)

def q8(x: torch.Tensor) -> torch.Tensor:
    """torch's E4M3 conversion (round to nearest even; finite for |x| <= 464) of fp64 values, via float32."""
    return x.float().to(torch.float8_e4m3fn).double()


def test_round_e4m3_matches_torch_conversion():
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double()
    vals = codes[torch.isfinite(codes)].unique().sort().values    # every finite E4M3 value
    mids = (vals[1:] + vals[:-1]) / 2                             # the ties, exact in float32
    rng = np.random.default_rng(3)
    wide = torch.from_numpy(rng.uniform(-464, 464, 20000)).float().double()
    small = torch.from_numpy(rng.uniform(-0.03, 0.03, 5000)).float().double()
    x = torch.cat([vals, mids, wide, small, torch.tensor([455.0, 464.0, -464.0])])
    np.testing.assert_array_equal(oracle.round_e4m3(x.numpy()), q8(x).numpy())
    assert oracle.round_e4m3([465.0, 1e6, -1e6]).tolist() == [448.0, 448.0, -448.0]  # saturating


def _eq15_step(m, l, o, s, v):
    """One iteration of the online softmax of Eq.15 over logits s [n] and values v [n, d] (torch, fp64)."""
    mi = torch.maximum(m, s.max())
    f = torch.exp(m - mi) if torch.isfinite(m) else torch.tensor(0.0, dtype=torch.float64)
    w = q8(256.0 * torch.exp(s - mi))
    return mi, l * f + w.sum(), o * f + w @ v


def test_eq15_one_iteration_is_the_quantised_softmax():
    # requests of at most one block: every tile runs one iteration (its diagonal block), so
    # O = sum P~ v / sum P~ and LSE = m + ln sum P~ - ln 256 with P~ = e4m3(2^8 e^{s - max s})
    w = small_workload(lengths=(128, 77), hq=8, hkv=2, dtype="e4m3")
    p = oracle.Problem.from_workload(w)
    res = oracle.run(p, alpha=0.0, sink=0, window=0, eq15=True)
    Q = dequant(p, p.q, p.c_q)
    for b in range(p.batch):
        s0, e0 = int(p.cu_seqlens[b]), int(p.cu_seqlens[b + 1])
        K, V = gathered(p, b)
        L = e0 - s0
        for hh in range(p.hq):
            logits = Q[s0:e0, hh] @ K[:, hh // p.g].T / math.sqrt(D)
            logits = logits.masked_fill(~torch.ones(L, L, dtype=torch.bool).tril(), float("-inf"))
            m = logits.max(-1, keepdim=True).values
            wts = q8(256.0 * torch.exp(logits - m))
            ref = (wts @ V[:, hh // p.g]) / wts.sum(-1, keepdim=True)
            assert rel_err(res["O"][s0:e0, hh], ref.numpy()) < 1e-12
            lse = m[:, 0] + torch.log(wts.sum(-1)) - math.log(256.0)
            np.testing.assert_allclose(res["lse"][s0:e0, hh], lse.numpy(), rtol=0, atol=1e-12)


def test_eq15_blocks_run_in_descending_order():
    # g = 1, one 256-token request, dense: tile 1 (positions 128..255) runs block 1, then block 0 (Eq.17). The
    # probabilities of block 1 are quantised against block 1's maximum and only rescaled when block 0 raises it;
    # the ascending order quantises differently, and the oracle must match the descending one only.
    w = small_workload(lengths=(256,), hq=1, hkv=1, dtype="e4m3", mu_scale=0.5, seed=4)
    p = oracle.Problem.from_workload(w)
    res = oracle.run(p, alpha=0.0, sink=0, window=0, eq15=True)
    Q = dequant(p, p.q, p.c_q)[:, 0]
    K, V = gathered(p, 0)
    K, V = K[:, 0], V[:, 0]
    worst_desc, best_asc = 0.0, 0.0
    for r in range(128, 256):
        s = Q[r] @ K[:r + 1].T / math.sqrt(D)
        out = []
        for order in ((1, 0), (0, 1)):
            m, l, o = torch.tensor(float("-inf"), dtype=torch.float64), torch.tensor(0.0, dtype=torch.float64), 0.0
            for J in order:
                sl = slice(128 * J, min(128 * J + 128, r + 1))
                m, l, o = _eq15_step(m, l, o, s[sl], V[sl])
            out.append((o / l).numpy())
        worst_desc = max(worst_desc, rel_err(res["O"][r, 0], out[0]))
        best_asc = max(best_asc, rel_err(res["O"][r, 0], out[1]))
    assert worst_desc < 1e-12
    assert best_asc > 1e-6


def test_eq15_correction_chunks_descending_with_operand_format_means():
    # g = 1, 130 blocks: the last tile (D = 129) appends its pruned blocks as two chunks of means, chunk 1
    # (block 128) before chunk 0 (blocks 0..127), each mean rounded to E4M3 with its tensor's scale and its
    # logit shifted by ln 128 (Eq.6). On these inputs chunk 0 raises the running maximum, so the chunk order
    # decides how chunk 1 is quantised: the ascending order must not match.
    w = small_workload(lengths=(130 * 128,), hq=1, hkv=1, dtype="e4m3", mu_scale=0.5, seed=6)
    p = oracle.Problem.from_workload(w)
    seg = oracle.segments(p)
    pooled = oracle.pool(p, seg)
    last = len(seg) - 1
    assert int(seg.D[last]) == 129
    sel = oracle.select(p, 0.05, 1, 0, seg=seg, pooled=pooled, seg_ids=[last])
    picked = sel.selected(seg, last)
    assert 128 not in picked and len(picked) < 100          # both chunks hold pruned blocks
    Ot, lt = oracle.attend(p, sel.sel_full, seg=seg, pooled=pooled, seg_ids=[last], eq15=True)
    Q = dequant(p, p.q, p.c_q)[:, 0]
    K, V = gathered(p, 0)
    K, V = K[:, 0], V[:, 0]
    # the operand-format means: the mean of each block's E4M3 codes (exact in fp64), rounded to E4M3 by the
    # encoder pinned above, times the tensor's scale
    kraw = torch.from_numpy(oracle.round_e4m3(K.numpy() / p.c_k)).reshape(130, 128, D)  # exact codes again
    vraw = torch.from_numpy(oracle.round_e4m3(V.numpy() / p.c_v)).reshape(130, 128, D)
    kop = torch.from_numpy(oracle.round_e4m3(kraw.mean(1).numpy())) * p.c_k
    vop = torch.from_numpy(oracle.round_e4m3(vraw.mean(1).numpy())) * p.c_v
    pruned = [J for J in range(129) if J not in set(picked.tolist())]
    worst_desc, best_asc = 0.0, 0.0
    for i in (0, 1, 64, 127):
        r = 129 * 128 + i
        s = Q[r] @ K[:r + 1].T / math.sqrt(D)
        res = []
        for chunks in ((1, 0), (0, 1)):
            m, l, o = torch.tensor(float("-inf"), dtype=torch.float64), torch.tensor(0.0, dtype=torch.float64), 0.0
            for J in sorted(picked.tolist(), reverse=True):
                sl = slice(128 * J, min(128 * J + 128, r + 1))
                m, l, o = _eq15_step(m, l, o, s[sl], V[sl])
            for chunk in chunks:
                Js = [J for J in pruned if J // 128 == chunk]
                sm = Q[r] @ kop[Js].T / math.sqrt(D) + math.log(128.0)
                m, l, o = _eq15_step(m, l, o, sm, vop[Js])
            res.append(((o / l).numpy(), float(m + torch.log(l) - math.log(256.0))))
        worst_desc = max(worst_desc, rel_err(Ot[0, i], res[0][0]))
        best_asc = max(best_asc, rel_err(Ot[0, i], res[1][0]))
        assert abs(lt[0, i] - res[0][1]) < 1e-12
    assert worst_desc < 1e-12
    assert best_asc > 1e-6


def test_eq15_stays_within_the_fp8_tolerance_of_the_exact_output():
    w = small_workload(lengths=(700, 300), hq=8, hkv=2, dtype="e4m3", mu_scale=0.7)
    p = oracle.Problem.from_workload(w)
    exact = oracle.run(p, alpha=0.2, sink=1, window=1)
    quant = oracle.run(p, alpha=0.2, sink=1, window=1, eq15=True)
    d = quant["O"] - exact["O"]
    rel_rms = float(np.sqrt((d ** 2).sum() / (exact["O"] ** 2).sum()))
    assert 1e-4 < rel_rms < 6e-2
    assert np.array_equal(quant["idx"], exact["idx"])        # the selection does not depend on the mode


# ------------------------------------------- Stage 2 integer work (visit order, correction masks, splits)

def _schedule_problem(length, page, permute, seed=3):
    """One request, one query head on one KV head (g = 1: tile t holds positions 128 t .. 128 t + 127, so its
    diagonal block is D = t); zero tensors, only the lengths and the page table matter."""
    q = np.zeros((length, 1, D), np.uint16)
    k = np.zeros((length, 1, D), np.uint16)
    return paged_problem(q, [k], [k], 1, 1, page=page, seed=seed, permute=permute)


def test_tile_schedule_hand_example():
    # D = 300, CSR {0, 5, 299, 300}: Eq.17 visits the selected blocks descending; todo = {J < 300} minus the
    # selected = {1..4, 6..298}; every 128-block chunk holds a todo block, visited 2, 1, 0
    p = _schedule_problem(128 * 301, page=64, permute=False)
    seg = oracle.segments(p)
    s = 300
    assert int(seg.D[s]) == 300
    cu = np.zeros(len(seg) + 1, np.int64)
    cu[s + 1:] = 4
    idx = np.array([0, 5, 299, 300])
    got = oracle.tile_schedule(p, seg, s, cu, idx)
    full = 0xffffffff
    want = [
        # identity page table of 64-token pages: block J's chunks start at rows 128 J and 128 J + 64
        (300, 0, 0, 0, 0, 38400, 38464),
        (299, 0, 0, 0, 0, 38272, 38336),
        (5, 0, 0, 0, 0, 640, 704),
        (0, 0, 0, 0, 0, 0, 64),
        # chunk 2: blocks 256..287 all pruned, 288..298 pruned (bits 0..10), 299 selected, nothing past D
        (-3, full, 0x7ff, 0, 0, 256, 0),
        (-2, full, full, full, full, 128, 0),
        # chunk 0: blocks 0 and 5 selected
        (-1, full & ~1 & ~(1 << 5), full, full, full, 0, 0),
    ]
    assert got.tolist() == [list(r) for r in want]
    # without correction: the four exact iterations only; dense mode: every block 300 .. 0
    assert oracle.tile_schedule(p, seg, s, cu, idx, correction=False)[:, 0].tolist() == [300, 299, 5, 0]
    dense = oracle.tile_schedule(p, seg, s, cu, idx, dense=True)
    assert dense[:, 0].tolist() == list(range(300, -1, -1))


def test_tile_schedule_page_rows_and_chunk_skipping():
    # 32-token pages through a permuted table: a block's first and last page chunks start at its tokens 128 J
    # and 128 J + 96. A chunk of means whose blocks are all selected is skipped.
    p = _schedule_problem(1000, page=32, permute=True, seed=11)
    seg = oracle.segments(p)
    s = len(seg) - 1
    D = int(seg.D[s])
    assert D == 7
    pt = p.page_table[0]
    cu = np.zeros(len(seg) + 1, np.int64)
    cu[s + 1:] = D + 1
    idx = np.arange(D + 1)       # every block selected: no correction chunk
    got = oracle.tile_schedule(p, seg, s, cu, idx)
    assert got[:, 0].tolist() == list(range(7, -1, -1))
    for row in got:
        J = int(row[0])
        assert row[5] == pt[4 * J] * 32 and row[6] == pt[4 * J + 3] * 32
    # the last block of the 1000-token request: its last page chunk (tokens 992..999) is page 31
    assert got[0, 6] == pt[31] * 32


def test_tile_schedule_out_of_range_chunk_row():
    # 130-token request with 16-token pages: block 1 holds tokens 128..129 only, so its last page chunk
    # (token 240) lies past the request and reads the pool's end row
    p = _schedule_problem(130, page=16, permute=False)
    seg = oracle.segments(p)
    s = 1
    assert int(seg.D[s]) == 1
    cu = np.array([0, 1, 3])
    idx = np.array([0, 0, 1])
    got = oracle.tile_schedule(p, seg, s, cu, idx)
    oob = p.k_pages.shape[0] * 16
    assert got[0].tolist() == [1, 0, 0, 0, 0, 128, oob]
    assert got[1].tolist() == [0, 0, 0, 0, 0, 0, 112]


def test_split_plan_closed_forms():
    # 4 tiles on 2 SMs (fewer than 4 x 2): C* = max(8, ceil(117 / 2)) = 59; the 100-iteration tile runs as
    # two runs of 50, the others whole
    target, runs = oracle.split_plan([100, 7, 7, 3], n_sms=2)
    assert target == 59
    assert runs == [[(0, 50), (50, 100)], [(0, 7)], [(0, 7)], [(0, 3)]]
    # 130 iterations against C* = 59: three runs of ceil(130 / 3) = 44, the last one shorter
    target, runs = oracle.split_plan([130, 1, 1, 1], n_sms=2)
    assert target == max(8, -(-133 // 2)) == 67
    assert runs[0] == [(0, 65), (65, 130)]
    # the floor of 8 iterations per run
    target, runs = oracle.split_plan([20, 1, 1], n_sms=152)
    assert target == 8 and runs[0] == [(0, 7), (7, 14), (14, 20)]
    # as many tiles as 4 x SMs: no splits
    target, runs = oracle.split_plan([1000] * 8, n_sms=2)
    assert target is None and all(r == [(0, 1000)] for r in runs)
