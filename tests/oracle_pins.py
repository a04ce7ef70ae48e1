"""Pins that tie the fp64 oracle to something other than itself.

Each ``check_*`` raises AssertionError when the oracle disagrees with: a closed form written
out here, the pages' worked views (``tests/golden``), the textbook complex-number form of RoPE,
torch's own scaled-dot-product attention, or the oracle's other (brute-force) formulation.
``test_oracle_pins.py`` runs them as they are; ``test_oracle_mutations.py`` plants plausible
mistakes in the oracle and checks that at least one of them fails.

Modules are looked up at call time (``R.rope``, ``A.method`` ...) so that a planted mistake
is seen.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle.attention as A
import oracle.cache as C
import oracle.rope as R

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------------------- RoPE


def rope_complex(x, pos, theta):
    """Textbook RoPE as complex multiplication: z_i = x_i + i x_{i+D/2}, z_i *= e^{i pos f_i}."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    f = np.array([theta ** (-(2.0 * i) / D) for i in range(h)])
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * np.asarray(pos, dtype=np.float64)[..., None] * f)
    return np.concatenate([z.real, z.imag], axis=-1)


def check_rope_complex_form():
    g = np.random.default_rng(11)
    for D, theta in ((2, 1e4), (8, 1e4), (64, 1e4), (128, 1e6)):
        x = g.standard_normal((7, D))
        pos = g.integers(-(1 << 17), 1 << 17, size=7)
        got = R.rope(x, pos, theta)
        ref = rope_complex(x, pos, theta)
        assert np.allclose(got, ref, rtol=0, atol=1e-9 * max(1.0, np.abs(ref).max())), (D, theta)


def check_rope_d2_textbook():
    # D = 2: one pair, f_0 = theta^0 = 1 rad per position: a plain 2-D rotation.
    for p in (0, 1, 2, -3, 1000):
        assert np.allclose(R.rope(np.array([1.0, 0.0]), p, 1e4), [math.cos(p), math.sin(p)], atol=1e-14)
        assert np.allclose(R.rope(np.array([0.0, 1.0]), p, 1e4), [-math.sin(p), math.cos(p)], atol=1e-14)


def check_inv_freq_values():
    f = R.inv_freq(64, 1e4)
    assert f[0] == 1.0
    assert abs(f[1] - 10 ** (-0.125)) < 1e-15          # 1e4^(-2/64)
    assert abs(f[31] - 10 ** (-4 * 62 / 64)) < 1e-18


def check_rope_invariants():
    """rho is orthogonal, composes additively, and q.k depends only on a - b."""
    g = np.random.default_rng(12)
    for D, theta in ((2, 1e4), (64, 1e4), (128, 1e6)):
        q, k = g.standard_normal(D), g.standard_normal(D)
        for _ in range(8):
            a, b, d = (int(x) for x in g.integers(-(1 << 17), 1 << 17, size=3))
            assert abs(np.linalg.norm(R.rope(q, a, theta)) - np.linalg.norm(q)) < 1e-12
            assert np.allclose(R.rope(R.rope(q, a, theta), b, theta), R.rope(q, a + b, theta), atol=1e-9)
            lhs = R.rope(q, a, theta) @ R.rope(k, b, theta)
            mid = R.rope(q, a - b, theta) @ k
            rhs = R.rope(q, a + d, theta) @ R.rope(k, b + d, theta)
            assert abs(lhs - mid) < 1e-9 and abs(lhs - rhs) < 1e-9


# ------------------------------------------------------------------------- cache views


def _tiny_cache(W=2, S=4, pages=64, H_kv=1, D=2, order=None, contiguous=False, layers=1):
    return C.HogwildCache(1, W, layers, H_kv, D, 1e4, S, pages, contiguous=contiguous,
                          page_order=order)


def _names_of_view(cache, p, w, names):
    entries, _ = cache.view(p, w)
    return [names[sid] for sid, _, _ in entries]


def check_views_golden():
    with open(os.path.join(GOLDEN, "views_w2.json")) as f:
        g2 = json.load(f)
    c = _tiny_cache(W=2)
    c.append(0, [[3, 2, 1]], np.ones((6, 1, 2)), np.ones((6, 1, 2)))
    names = {c.common[0][0]: "C", c.live[0][0]: "A", c.live[0][1]: "B"}
    assert _names_of_view(c, 0, 0, names) == g2["views"]["A"]
    assert _names_of_view(c, 0, 1, names) == g2["views"]["B"]
    with open(os.path.join(GOLDEN, "views_ordering_w4.json")) as f:
        g4 = json.load(f)
    c = _tiny_cache(W=4)
    c.append(0, [[2, 1, 1, 1, 1]], np.ones((6, 1, 2)), np.ones((6, 1, 2)))
    names = {c.common[0][0]: "C"}
    names.update({c.live[0][w]: f"W{w}" for w in range(4)})
    for w in range(4):
        assert _names_of_view(c, 0, w, names) == g4["views"][f"W{w}"]


def check_view_offsets_and_query_position():
    # Append happens before attention (inference flow): the own block includes this step's
    # token and the query is the last position of the view; offsets are running sums.
    c = _tiny_cache(W=2)
    c.append(0, [[5, 3, 2]], np.ones((10, 1, 2)), np.ones((10, 1, 2)))
    entries, i_q = c.view(0, 0)
    assert [(off, n) for _, off, n in entries] == [(0, 5), (5, 2), (7, 3)] and i_q == 9
    entries, i_q = c.view(0, 1)
    assert [(off, n) for _, off, n in entries] == [(0, 5), (5, 3), (8, 2)] and i_q == 9


def check_pages_hand_example():
    """Deterministic FIFO page allocation, worked by hand (page size 4)."""
    c = _tiny_cache(W=2, S=4, pages=8, order=[5, 2, 7, 0, 1, 3, 4, 6])
    z = lambda n: np.zeros((n, 1, 2))
    c.append(0, [[5, 3, 0]], z(8), z(8))        # common j=0..4 -> 5, 2 ; w0 j=0..2 -> 7
    c.step_end([[0, 0]])
    t = c.tables()
    assert [s[4] for s in t["segments"]] == [[5, 2], [7], []]
    c.append(0, [[0, 1, 1]], z(2), z(2))        # w0 j=3: none ; w1 j=0 -> 0
    c.step_end([[1, 0]])                        # w0 commits: its block joins the common list
    t = c.tables()
    assert t["common"] == [[0, 1]] and t["live"] == [[3, 2]]
    assert [s[2] for s in t["segments"]] == [5, 4, 1, 0]
    c.append(0, [[2, 1, 1]], z(4), z(4))        # common tail = seg1 j=4,5 -> 1 ; seg3 j=0 -> 3
    t = c.tables()
    assert [s[4] for s in t["segments"]] == [[5, 2], [7, 1], [0], [3]]
    assert t["free_count"] == 2
    e0, q0 = c.view(0, 0)
    e1, q1 = c.view(0, 1)
    assert [(s, o, n) for s, o, n in e0] == [(0, 0, 5), (1, 5, 6), (2, 11, 2), (3, 13, 1)] and q0 == 13
    assert [(s, o, n) for s, o, n in e1] == [(0, 0, 5), (1, 5, 6), (3, 11, 1), (2, 12, 2)] and q1 == 13
    c.step_end([[0, 0]])
    c.append(0, [[9, 0, 0]], z(9), z(9))        # seg1 j=6..14: pages at j=8 -> 4, j=12 -> 6
    c.step_end([[0, 0]])
    c.append(0, [[1, 0, 0]], z(1), z(1))        # j=15: no new page
    c.step_end([[0, 0]])
    before = c.tables()
    assert before["free_count"] == 0 and before["segments"][1][4] == [7, 1, 4, 6]
    try:
        c.append(0, [[1, 0, 0]], z(1), z(1))    # j=16 needs a page and none is left
        raise AssertionError("expected OutOfPages")
    except C.OutOfPages:
        pass
    assert c.tables() == before                 # a refused append changes nothing


def check_simultaneous_commits_in_ascending_id():
    """Workers that finish in the same step join the common history in ascending id, each
    keeping its pages; fresh blocks get new segment ids in the same order."""
    c = _tiny_cache(W=3, S=4, pages=16)
    z = lambda n: np.zeros((n, 1, 2))
    c.append(0, [[2, 1, 2, 3]], z(8), z(8))
    c.step_end([[1, 0, 1]])
    t = c.tables()
    assert t["common"] == [[0, 1, 3]] and t["live"] == [[4, 2, 5]]
    e, i_q = c.view(0, 1)
    assert [(s, o, n) for s, o, n in e] == [(0, 0, 2), (1, 2, 1), (3, 3, 3), (2, 6, 2)] and i_q == 7


# ----------------------------------------------------------------- worked 2-worker example


def _two_worker_d2(k_vec):
    """C=[c0], A=[a0], B=[b0]; D=2, H=1; q=(1,0); every raw key = k_vec.
    Values: v_C=(1,0), v_A=(0,0), v_B=(0,1), so out reads off the softmax weights."""
    c = _tiny_cache(W=2, S=4)
    k = np.array([k_vec, k_vec, k_vec], dtype=np.float64).reshape(3, 1, 2)
    v = np.array([[1.0, 0.0], [0.0, 0.0], [0.0, 1.0]]).reshape(3, 1, 2)   # order C, A, B
    c.append(0, [[1, 1, 1]], k, v)
    q = np.array([1.0, 0.0]).reshape(1, 1, 1, 2).repeat(2, axis=1)
    return c, q


def check_two_worker_hand(fn_name="method"):
    fn = getattr(A, fn_name)
    r2 = 1.0 / math.sqrt(2.0)
    for k_vec, raw in (((1.0, 0.0), (math.cos(2), math.cos(1), 1.0)),
                       ((0.0, 1.0), (math.sin(2), math.sin(1), 0.0))):
        c, q = _two_worker_d2(k_vec)
        out, lse = fn(c, 0, q)
        s = [x * r2 for x in raw]                  # scores at view positions 0, 1, 2 (i_q = 2)
        e = [math.exp(x) for x in s]
        w = [x / sum(e) for x in e]
        # Alice (worker 0) sees C, B, A: out = w0 v_C + w1 v_B + w2 v_A = (w0, w1)
        assert np.allclose(out[0, 0, 0], [w[0], w[1]], atol=1e-13), (k_vec, out[0, 0, 0], w)
        # Bob (worker 1) sees C, A, B: out = w0 v_C + w1 v_A + w2 v_B = (w0, w2)
        assert np.allclose(out[0, 1, 0], [w[0], w[2]], atol=1e-13), (k_vec, out[0, 1, 0], w)
        assert abs(lse[0, 0, 0] - math.log(sum(e))) < 1e-13


# --------------------------------------------------------------- random brute vs method


def random_session(seed, D, W, H_kv=2, G=2, S=4, steps=4, P=2, commit_p=0.5, maxlen=40):
    """Random cache history with appends to every block and random commits.

    Yields (cache, q) after each step's append (before step_end)."""
    g = np.random.default_rng(seed)
    c = C.HogwildCache(P, W, 1, H_kv, D, 1e4 if D <= 64 else 1e6, S, 4096,
                       page_order=g.permutation(4096))
    Hq = H_kv * G
    for step in range(steps):
        if step == 0:
            n = g.integers(0, maxlen + 1, size=(P, W + 1))
        else:
            n = g.integers(0, 4, size=(P, W + 1))
        tot = int(n.sum())
        c.append(0, n, g.standard_normal((tot, H_kv, D)), g.standard_normal((tot, H_kv, D)))
        q = g.standard_normal((P, W, Hq, D))
        yield c, q
        c.step_end((g.random((P, W)) < commit_p).astype(np.uint8))


def check_brute_vs_method(seeds=range(6)):
    for seed in seeds:
        for D in (2, 4, 64):
            W = 1 + seed % 4
            for c, q in random_session(seed, D, W):
                ob, lb = A.brute_force(c, 0, q)
                om, lm = A.method(c, 0, q)
                assert np.allclose(ob, om, rtol=0, atol=1e-10), (seed, D, np.abs(ob - om).max())
                fin = np.isfinite(lb)
                assert (fin == np.isfinite(lm)).all()
                assert np.allclose(lb[fin], lm[fin], rtol=0, atol=1e-10)


# ------------------------------------------------------------------------- closed forms


def check_zero_keys_give_mean_values():
    g = np.random.default_rng(13)
    for c, q in random_session(21, 64, 3, steps=2):
        for seg in c.segments:
            for lst in (seg._raw_k[0], seg._stored_k[0]):
                for a in lst:
                    a[:] = 0.0
            seg._cat.clear()
        for fn in (A.brute_force, A.method):
            out, _ = fn(c, 0, q)
            for p in range(c.P):
                for w in range(c.W):
                    entries, _ = c.view(p, w)
                    if not entries:
                        continue
                    v = np.concatenate([c.segments[s].raw_v(0)[:n] for s, _, n in entries])
                    for h in range(q.shape[2]):
                        assert np.allclose(out[p, w, h], v[:, h // 2].mean(axis=0), atol=1e-12)
    del g


def check_single_token_returns_its_value():
    c = _tiny_cache(W=1, S=4, H_kv=1, D=64)
    g = np.random.default_rng(14)
    v = g.standard_normal((1, 1, 64))
    c.append(0, [[0, 1]], g.standard_normal((1, 1, 64)), v)
    for fn in (A.brute_force, A.method):
        out, lse = fn(c, 0, g.standard_normal((1, 1, 3, 64)))
        assert np.allclose(out[0, 0], v[0, 0], atol=1e-14)


def check_single_worker_is_textbook_decode():
    """W = 1: the view is the common block then the own block, i.e. ordinary RoPE decode.
    Compare with torch's scaled_dot_product_attention on keys rotated by the complex form."""
    import torch
    g = np.random.default_rng(15)
    D, H_kv, G, theta = 64, 2, 3, 1e4
    c = C.HogwildCache(1, 1, 1, H_kv, D, theta, 8, 256)
    k0, v0 = g.standard_normal((23, H_kv, D)), g.standard_normal((23, H_kv, D))
    c.append(0, [[17, 6]], k0, v0)
    c.step_end([[0]])
    k1, v1 = g.standard_normal((1, H_kv, D)), g.standard_normal((1, H_kv, D))
    c.append(0, [[0, 1]], k1, v1)
    q = g.standard_normal((1, 1, H_kv * G, D))
    kk = np.concatenate([k0, k1])
    vv = np.concatenate([v0, v1])
    n = kk.shape[0]
    krot = rope_complex(kk, np.arange(n)[:, None], theta)          # [n][H_kv][D]
    qrot = rope_complex(q[0, 0], n - 1, theta)                      # [H_q][D]
    kt = torch.from_numpy(np.repeat(krot.transpose(1, 0, 2), G, axis=0))   # [H_q][n][D]
    vt = torch.from_numpy(np.repeat(vv.transpose(1, 0, 2), G, axis=0))
    qt = torch.from_numpy(qrot[:, None, :])                         # [H_q][1][D]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt).numpy()[:, 0, :]
    for fn in (A.brute_force, A.method):
        out, _ = fn(c, 0, q)
        assert np.allclose(out[0, 0], ref, atol=1e-12), np.abs(out[0, 0] - ref).max()


def check_relabel_two_workers():
    """Swapping the two workers' data swaps their outputs (C+B+A <-> C+A+B)."""
    g = np.random.default_rng(16)
    D, H_kv = 64, 1
    kc, vc = g.standard_normal((9, H_kv, D)), g.standard_normal((9, H_kv, D))
    ka, va = g.standard_normal((4, H_kv, D)), g.standard_normal((4, H_kv, D))
    kb, vb = g.standard_normal((6, H_kv, D)), g.standard_normal((6, H_kv, D))
    qa, qb = g.standard_normal((2, D)), g.standard_normal((2, D))
    c1 = C.HogwildCache(1, 2, 1, H_kv, D, 1e4, 8, 64)
    c1.append(0, [[9, 4, 6]], np.concatenate([kc, ka, kb]), np.concatenate([vc, va, vb]))
    c2 = C.HogwildCache(1, 2, 1, H_kv, D, 1e4, 8, 64)
    c2.append(0, [[9, 6, 4]], np.concatenate([kc, kb, ka]), np.concatenate([vc, vb, va]))
    o1, _ = A.method(c1, 0, np.stack([qa, qb])[None])
    o2, _ = A.method(c2, 0, np.stack([qb, qa])[None])
    assert np.allclose(o1[0, 0], o2[0, 1], atol=1e-13) and np.allclose(o1[0, 1], o2[0, 0], atol=1e-13)


# ------------------------------------------------------------------------- cache layouts


def _layout_scenario(layout, D=2, H_kv=1, seed=None):
    """The hand-worked scenario of views_layouts_w3.json: prompt 4, A 2, B 1, C 3; A commits;
    then one token for every worker.  Returns the cache and the block -> segment id names."""
    g = np.random.default_rng(seed)
    draw = (lambda n: g.standard_normal((n, H_kv, D))) if seed is not None else \
        (lambda n: np.ones((n, H_kv, D)))
    c = C.HogwildCache(1, 3, 1, H_kv, D, 1e4, 4, 64, layout=layout)
    c.append(0, [[4, 2, 1, 3]], draw(10), draw(10))
    c.step_end([[1, 0, 0]])
    c.append(0, [[0, 1, 1, 1]], draw(3), draw(3))
    names = {c.common[0][0]: "P", c.common[0][1]: "A1", c.live[0][0]: "A2", c.live[0][1]: "B",
             c.live[0][2]: "C"}
    return c, names


def check_layout_views_golden():
    with open(os.path.join(GOLDEN, "views_layouts_w3.json")) as f:
        gl = json.load(f)
    for layout, views in gl["views"].items():
        c, names = _layout_scenario(layout)
        for w, who in enumerate("ABC"):
            entries, i_q = c.view(0, w)
            got = [[names[sid], off] for sid, off, n in entries]
            assert got == views[who], (layout, who, got)
            assert [n for _, _, n in entries] == [gl["lengths"][b] for b, _ in views[who]]
            assert i_q == gl["i_q"][layout][who], (layout, who, i_q)


def check_layouts_textbook_attention():
    """Every layout: the method equals textbook RoPE attention over the golden's block order
    (raw keys laid out at positions 0 .. n-1, rotated by the complex form, query at i_q)."""
    with open(os.path.join(GOLDEN, "views_layouts_w3.json")) as f:
        gl = json.load(f)
    D, H_kv, G, theta = 8, 2, 2, 1e4
    q = np.random.default_rng(31).standard_normal((1, 3, H_kv * G, D))
    for layout, views in gl["views"].items():
        c, names = _layout_scenario(layout, D=D, H_kv=H_kv, seed=30)
        by_name = {v: k for k, v in names.items()}
        out, lse = A.method(c, 0, q)
        for w, who in enumerate("ABC"):
            blocks = [b for b, _ in views[who]]
            kr = np.concatenate([c.segments[by_name[b]].raw_k(0) for b in blocks])
            vr = np.concatenate([c.segments[by_name[b]].raw_v(0) for b in blocks])
            n = kr.shape[0]
            k = rope_complex(kr, np.arange(n)[:, None], theta)
            qr = rope_complex(q[0, w], gl["i_q"][layout][who], theta)
            for h in range(H_kv * G):
                sc = k[:, h // G, :] @ qr[h] / math.sqrt(D)
                e = np.exp(sc - sc.max())
                ref = e @ vr[:, h // G, :] / e.sum()
                assert np.allclose(out[0, w, h], ref, atol=1e-12), (layout, who, h)
                assert abs(lse[0, w, h] - (sc.max() + math.log(e.sum()))) < 1e-12


def check_layouts_coincide_without_commits():
    """With no commit yet, the prompt is the whole common history: contiguous equals combined
    and no-sync equals step-wise (section 6: the layouts differ only in how finished and
    unfinished steps are shared)."""
    g = np.random.default_rng(32)
    k, v = g.standard_normal((14, 1, 8)), g.standard_normal((14, 1, 8))
    caches = {}
    for layout in C.LAYOUTS:
        c = C.HogwildCache(1, 3, 1, 1, 8, 1e4, 4, 64, layout=layout)
        c.append(0, [[5, 3, 4, 2]], k, v)
        caches[layout] = c
    for w in range(3):
        assert caches["contiguous"].view(0, w) == caches["combined"].view(0, w)
        assert caches["no_sync"].view(0, w) == caches["step_wise"].view(0, w)
        assert [s for s, _, _ in caches["step_wise"].view(0, w)[0]] == \
            [caches["step_wise"].common[0][0], caches["step_wise"].live[0][w]]


# ------------------------------------------------------------- several queries per worker


def _mq_counts(g, c):
    """A random query count per worker: at most its own block's visible length (0 if empty)."""
    n_q = np.zeros((c.P, c.W), dtype=np.int64)
    for p in range(c.P):
        for w in range(c.W):
            n = c.segments[c.live[p][w]].visible
            n_q[p, w] = g.integers(0, min(n, 5) + 1) if n else 0
    return n_q


def check_mq_brute_vs_method():
    """The two causal formulations agree, over random histories, commits and every layout."""
    for seed in range(4):
        g = np.random.default_rng(100 + seed)
        for layout in C.LAYOUTS:
            for c, _ in random_session(seed, 8, 1 + seed % 3, P=2):
                c.layout = layout
                n_q = _mq_counts(g, c)
                q = g.standard_normal((int(n_q.sum()), 4, 8))
                ob, lb = A.brute_force_mq(c, 0, q, n_q)
                om, lm = A.method_mq(c, 0, q, n_q)
                assert np.allclose(ob, om, rtol=0, atol=1e-10), (seed, layout)
                assert np.allclose(lb, lm, rtol=0, atol=1e-10)


def check_mq_one_query_is_decode():
    """One query per worker is the decode step: method_mq equals method row for row."""
    g = np.random.default_rng(110)
    tried = 0
    for c, q in random_session(7, 8, 3, P=2, commit_p=0.0):
        ok = all(c.segments[c.live[p][w]].visible > 0 for p in range(c.P) for w in range(c.W))
        if not ok:
            continue
        tried += 1
        n_q = np.ones((c.P, c.W), dtype=np.int64)
        om, lm = A.method_mq(c, 0, q.reshape(-1, q.shape[2], q.shape[3]), n_q)
        od, ld = A.method(c, 0, q)
        assert np.allclose(om, od.reshape(om.shape), rtol=0, atol=1e-12)
        assert np.allclose(lm, ld.reshape(lm.shape), rtol=0, atol=1e-12)
    assert tried >= 2
    del g


def check_mq_chunk_equals_token_by_token():
    """Query token t of a chunk sees what a single decode query sees when the worker's block
    ends at that token (the cache rebuilt with the block cut there)."""
    g = np.random.default_rng(111)
    D, H_kv, W = 8, 2, 3
    lens = [6, 2, 5, 3]                      # common, workers 0..2
    tot = sum(lens)
    k, v = g.standard_normal((tot, H_kv, D)), g.standard_normal((tot, H_kv, D))
    c = C.HogwildCache(1, W, 1, H_kv, D, 1e4, 4, 64)
    c.append(0, [lens], k, v)
    n_q = np.array([[0, 4, 2]])
    q = g.standard_normal((6, 2 * H_kv, D))
    out, lse = A.method_mq(c, 0, q, n_q)
    starts = np.cumsum([0] + lens)
    i = 0
    for w in range(W):
        for t in range(int(n_q[0, w])):
            cut = lens[1 + w] - (int(n_q[0, w]) - 1 - t)
            sub = [lens[0]] + [lens[1 + u] if u != w else cut for u in range(W)]
            keep = np.concatenate([np.arange(starts[b], starts[b] + sub[b]) for b in range(W + 1)])
            c2 = C.HogwildCache(1, W, 1, H_kv, D, 1e4, 4, 64)
            c2.append(0, [sub], k[keep], v[keep])
            qd = np.zeros((1, W, 2 * H_kv, D))
            qd[0, w] = q[i]
            od, ld = A.method(c2, 0, qd)
            assert np.allclose(out[i], od[0, w], rtol=0, atol=1e-12), (w, t)
            assert np.allclose(lse[i], ld[0, w], rtol=0, atol=1e-12)
            i += 1


def check_mq_single_worker_is_causal_prefill():
    """W = 1 with a chunk of n queries is ordinary causal RoPE attention over prompt + block:
    torch's scaled_dot_product_attention with a lower-triangular mask on complex-form RoPE."""
    import torch
    g = np.random.default_rng(112)
    D, H_kv, G, theta, nq = 64, 2, 2, 1e4, 5
    c = C.HogwildCache(1, 1, 1, H_kv, D, theta, 8, 256)
    k, v = g.standard_normal((19, H_kv, D)), g.standard_normal((19, H_kv, D))
    c.append(0, [[12, 7]], k, v)
    q = g.standard_normal((nq, H_kv * G, D))
    n = 19
    pos_q = np.arange(n - nq, n)
    kr = rope_complex(k, np.arange(n)[:, None], theta)
    qr = np.stack([rope_complex(q[t], pos_q[t], theta) for t in range(nq)])    # [nq][H_q][D]
    kt = torch.from_numpy(np.repeat(kr.transpose(1, 0, 2), G, axis=0))        # [H_q][n][D]
    vt = torch.from_numpy(np.repeat(v.transpose(1, 0, 2), G, axis=0))
    qt = torch.from_numpy(qr.transpose(1, 0, 2).copy())                        # [H_q][nq][D]
    mask = torch.from_numpy(np.arange(n)[None, :] <= pos_q[:, None])
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask).numpy()
    out, _ = A.method_mq(c, 0, q, [[nq]])
    assert np.allclose(out, ref.transpose(1, 0, 2), atol=1e-12), np.abs(out - ref.transpose(1, 0, 2)).max()


# ------------------------------------------------------------------------- compaction


def _compaction_history(seed, layout="combined", S=4):
    g = np.random.default_rng(seed)
    c = C.HogwildCache(1, 3, 2, 2, 8, 1e4, S, 64, layout=layout, page_order=g.permutation(64))
    for n, fin in (([[5, 3, 2, 4]], [[1, 0, 1]]), ([[1, 2, 1, 1]], [[0, 1, 0]]),
                   ([[0, 2, 3, 1]], [[1, 1, 0]])):
        tot = int(np.sum(n))
        for layer in range(2):
            c.append(layer, n, g.standard_normal((tot, 2, 8)), g.standard_normal((tot, 2, 8)))
        c.step_end(fin)
    return c, g


def _next_step(c, g):
    for layer in range(2):
        c.append(layer, [[1, 1, 1, 1]], g.standard_normal((4, 2, 8)), g.standard_normal((4, 2, 8)))
    return g.standard_normal((1, 3, 4, 8))


def check_compaction_keeps_outputs():
    """Re-rotating committed segments into one frame (reading 1) and keeping them in their own
    frames with the offset absorbed by the query (reading 2) give the same attention."""
    import copy
    for layout in ("combined", "step_wise"):
        for first, count in ((0, 2), (1, 3), (0, 6), (2, 2)):
            c, g = _compaction_history(40 + first + count, layout)
            c2 = copy.deepcopy(c)
            c2.compact(0, first, count)
            q = _next_step(c, copy.deepcopy(g))
            q2 = _next_step(c2, g)
            assert np.array_equal(q, q2)
            for layer in range(2):
                o1, l1 = A.method(c, layer, q)
                o2, l2 = A.method(c2, layer, q2)
                ob, lb = A.brute_force(c2, layer, q2)
                assert np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1, l2, atol=1e-12)
                assert np.allclose(o2, ob, rtol=0, atol=1e-12)


def check_compaction_rerotates_stored_keys():
    """The merged keys are the old stored keys turned by their segment's offset in the merge
    (the rotation composes additively: rho(rho(k, j), o) = rho(k, j + o))."""
    c, _ = _compaction_history(50)
    olds = [c.segments[s] for s in c.common[0][1:4]]
    offs = np.cumsum([0] + [s.length for s in olds])
    expect = np.concatenate([rope_complex(s.stored_k(1), offs[i], 1e4)
                             for i, s in enumerate(olds) if s.length])
    sid = c.compact(0, 1, 3)
    assert np.allclose(c.segments[sid].stored_k(1), expect, rtol=0, atol=1e-12)


def check_compaction_pages_hand():
    """Worked by hand, page size 4: prompt 5 (pages 9, 8), A's paragraph 3 (page 7), B's 6
    (pages 6, 5).  Merging all three (14 tokens) takes the next four free pages 4, 3, 2, 1; the
    old pages return to the end of the free list as 9, 8, 7, 6, 5."""
    c = C.HogwildCache(1, 2, 1, 1, 2, 1e4, 4, 10, page_order=list(range(9, -1, -1)))
    c.append(0, [[5, 3, 6]], np.ones((14, 1, 2)), np.ones((14, 1, 2)))
    c.step_end([[1, 1]])
    t = c.tables()
    assert [s[4] for s in t["segments"][:3]] == [[9, 8], [7], [6, 5]]
    assert t["free_count"] == 5
    sid = c.compact(0, 0, 3)
    t = c.tables()
    assert sid == 5 and t["common"] == [[5]]
    assert t["segments"][5] == (0, -1, 14, 0, [4, 3, 2, 1])
    assert [s[2:] for s in t["segments"][:3]] == [(0, 0, [])] * 3
    assert list(c.free) == [0, 9, 8, 7, 6, 5]
    entries, i_q = c.view(0, 0)
    assert entries[0] == (5, 0, 14)


def check_compaction_refusals():
    c, _ = _compaction_history(60, "contiguous")
    try:
        c.compact(0, 1, 2)              # A's and C's paragraphs: two writers
        raise AssertionError("mixed writers merged in the contiguous layout")
    except C.InvalidArg:
        pass
    c.append(0, [[1, 1, 1, 1]], np.ones((4, 2, 8)), np.ones((4, 2, 8)))
    try:
        c.compact(0, 0, 2)
        raise AssertionError("compaction during a step")
    except C.InvalidArg:
        pass


# ------------------------------------------------------------- split over KV entries


def _random_ranges(g, total, k):
    """k ranges that partition [0, total) at random cut points (some of them empty)."""
    cuts = np.sort(g.integers(0, total + 1, size=k - 1)) if k > 1 else np.array([], int)
    edges = np.concatenate([[0], cuts, [total]]).astype(int)
    return [(int(edges[i]), int(edges[i + 1])) for i in range(k)]


def check_range_brute_vs_method(seeds=range(4)):
    """The method over selected entries (per-segment query rotation, LSE merge) against the
    plain definition (every key re-rotated at its view position, softmax over the selected
    keys), for random histories with commits and ranges cutting segments anywhere."""
    for seed in seeds:
        g = np.random.default_rng(100 + seed)
        for D in (2, 64):
            for c, q in random_session(seed, D, 1 + seed % 4):
                tot = [A.entry_spans(c, p)[1] for p in range(c.P)]
                for _ in range(3):
                    rg = []
                    for t in tot:
                        b = int(g.integers(0, t + 1))
                        rg.append((b, int(g.integers(b, t + 1))))
                    ob, lb = A.brute_force_range(c, 0, q, rg)
                    om, lm = A.method_range(c, 0, q, rg)
                    assert np.allclose(ob, om, rtol=0, atol=1e-10), (seed, D, rg)
                    fin = np.isfinite(lb)
                    assert (fin == np.isfinite(lm)).all()
                    assert np.allclose(lb[fin], lm[fin], rtol=0, atol=1e-10)


def check_range_partition_merges_to_full(seeds=range(4)):
    """Results over ranges that partition every problem's entries, merged by log-sum-exp,
    equal the attention over the whole view (the brute-force definition, pinned above)."""
    for seed in seeds:
        g = np.random.default_rng(200 + seed)
        for D in (2, 64):
            for c, q in random_session(seed, D, 1 + seed % 4):
                tot = [A.entry_spans(c, p)[1] for p in range(c.P)]
                k = int(g.integers(1, 5))
                per = [_random_ranges(g, t, k) for t in tot]
                parts = [A.method_range(c, 0, q, [per[p][i] for p in range(c.P)]) for i in range(k)]
                out, lse = A.merge_parts([o for o, _ in parts], [l for _, l in parts])
                ob, lb = A.brute_force(c, 0, q)
                assert np.allclose(out, ob, rtol=0, atol=1e-10), (seed, D, k)
                fin = np.isfinite(lb)
                assert (fin == np.isfinite(lse)).all()
                assert np.allclose(lse[fin], lb[fin], rtol=0, atol=1e-10)


def check_range_selects_segment_order_hand():
    """Entries are numbered common first, then the workers' blocks by id, whatever the view:
    prompt C (3 tokens) = entries 0-2, Alice's block (2) = 3-4, Bob's (2) = 5-6.  With all
    keys zero every score is 0, so a worker's output is the mean of the selected values and
    lse = log(count), for both workers alike."""
    c = _tiny_cache(W=2, S=4, pages=32, H_kv=1, D=2)
    n = np.array([[3, 2, 2]])
    vals = np.array([[10.0, 0.0], [20.0, 0.0], [30.0, 0.0],      # prompt
                     [1.0, 0.0], [0.0, 1.0],                     # Alice
                     [5.0, 5.0], [7.0, 9.0]])                    # Bob
    c.append(0, n, np.zeros((7, 1, 2)), vals[:, None, :])
    q = np.array([[[[0.3, -0.2]], [[1.1, 0.4]]]])
    for (b, e), mean in (((3, 5), [0.5, 0.5]), ((5, 7), [6.0, 7.0]), ((2, 4), [15.5, 0.0]),
                         ((0, 3), [20.0, 0.0]), ((4, 6), [2.5, 3.0])):
        for fn in (A.method_range, A.brute_force_range):
            out, lse = fn(c, 0, q, [(b, e)])
            for w in range(2):
                assert np.allclose(out[0, w, 0], mean, atol=1e-13), (fn.__name__, b, e, w, out[0, w, 0])
                assert abs(lse[0, w, 0] - math.log(e - b)) < 1e-13
    out, lse = A.method_range(c, 0, q, [(4, 4)])
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def check_merge_parts_closed_form():
    """Two parts with sums of exponentials 1 and 3 (lse 0 and log 3): weights 1/4 and 3/4, and
    merged lse log 4; an empty part (lse -inf) changes nothing; all parts empty give 0, -inf."""
    a, b = np.array([[2.0, -4.0]]), np.array([[6.0, 8.0]])
    out, lse = A.merge_parts([a, b], [np.array([0.0]), np.array([math.log(3.0)])])
    assert np.allclose(out, [[5.0, 5.0]], atol=1e-14) and abs(lse[0] - math.log(4.0)) < 1e-14
    out2, lse2 = A.merge_parts([a, b, np.full((1, 2), 99.0)],
                               [np.array([0.0]), np.array([math.log(3.0)]), np.array([-np.inf])])
    assert np.allclose(out2, out, atol=1e-14) and abs(lse2[0] - lse[0]) < 1e-14
    out3, lse3 = A.merge_parts([a, b], [np.array([-np.inf]), np.array([-np.inf])])
    assert np.all(out3 == 0) and np.isneginf(lse3[0])


ALL_CHECKS = [
    check_rope_complex_form, check_rope_d2_textbook, check_inv_freq_values, check_rope_invariants,
    check_views_golden, check_view_offsets_and_query_position, check_pages_hand_example,
    check_simultaneous_commits_in_ascending_id,
    check_two_worker_hand, check_brute_vs_method, check_zero_keys_give_mean_values,
    check_single_token_returns_its_value, check_single_worker_is_textbook_decode,
    check_relabel_two_workers, check_layout_views_golden, check_layouts_textbook_attention,
    check_layouts_coincide_without_commits, check_mq_brute_vs_method, check_mq_one_query_is_decode,
    check_mq_chunk_equals_token_by_token, check_mq_single_worker_is_causal_prefill,
    check_compaction_keeps_outputs, check_compaction_rerotates_stored_keys,
    check_compaction_pages_hand, check_compaction_refusals,
    check_range_brute_vs_method, check_range_partition_merges_to_full,
    check_range_selects_segment_order_hand, check_merge_parts_closed_form,
]
