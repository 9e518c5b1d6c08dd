"""CPU checks of the C ABI: the library loads and exports every declared symbol, the host-side
packing matches the oracle bit for bit, and bad arguments are rejected before any launch."""
import ctypes as C
import os
import re

import pytest
import torch

from oracle import prefix_grouper_oracle as orc
from shared_prefix_grouped_gb300 import _lib, api, flops
from shared_prefix_grouped_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    build()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(pg_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert "pg_grouped_attn_fwd" in names and "pg_pack" in names
    handle = C.CDLL(_lib.LIB_PATH)
    for n in names:
        assert hasattr(handle, n), n
    assert set(names) <= set(_lib.SIGNATURES)


TOK_CASES = [
    ([3, 2], [2, 3], [2, 1, 1, 0, 2]),
    ([0], [3], [5, 0, 2]),
    ([7], [0], []),
    ([130, 0, 64], [3, 2, 1], [1, 200, 63, 65, 0, 128]),
    ([300], [4], [64, 1, 127, 129]),
]


def expand_mask(tok):
    """Visibility implied by the library's per-token table {g0, pe, own_lo, pos}."""
    T = tok.shape[0]
    t = torch.arange(T)[:, None]
    s = torch.arange(T)[None, :]
    g0, pe, own = tok[:, 0:1], tok[:, 1:2], tok[:, 2:3]
    return (s <= t) & (s >= g0) & ((s < pe) | (s >= own))


def unpack(tab, struct):
    T = struct.total_tokens
    raw = tab.numpy().tobytes()
    tok = torch.frombuffer(bytearray(raw[struct.off_tokens: struct.off_tokens + 16 * T]),
                           dtype=torch.int32).view(T, 4).clone()
    lists = []
    for w in range(6):
        n = struct.n_tiles[w]
        o = struct.off_tiles[w]
        lists.append(torch.frombuffer(bytearray(raw[o: o + 32 * n]), dtype=torch.int32)
                     .view(n, 8).clone() if n else torch.zeros((0, 8), dtype=torch.int32))
    return tok, lists


@pytest.mark.parametrize("case", TOK_CASES)
def test_pack_host_matches_oracle_bit_exactly(case):
    plens, gsz, rs = case
    pos, tab, st = api.pack_host(plens, gsz, rs)
    lay = orc.pack_layout(plens, gsz, rs)
    assert st.total_tokens == lay.total_tokens
    assert torch.equal(pos.to(torch.int64), lay.position_ids)
    tok, lists = unpack(tab, st)
    assert torch.equal(tok[:, 3].to(torch.int64), lay.position_ids)
    mask = orc.visibility_mask(lay)
    assert torch.equal(expand_mask(tok), mask)
    assert st.pairs == int(mask.sum()) == flops.total_pairs(plens, gsz, rs)
    T = lay.total_tokens
    for w, bm in [(0, 64), (1, 128), (4, 256)]:
        ft = lists[w]
        # forward tiles: cover every row once; their key ranges cover every visible key
        covered = torch.zeros(T, dtype=torch.int32)
        for q0, q1, g0, p_end, s_lo, s_hi, pe, _ in ft.tolist():
            assert 0 < q1 - q0 <= bm
            covered[q0:q1] += 1
            keys = torch.zeros(T, dtype=torch.bool)
            keys[g0:p_end] = True
            keys[s_lo:s_hi] = True
            assert not bool((mask[q0:q1] & ~keys[None, :]).any())
        assert torch.equal(covered, torch.ones(T, dtype=torch.int32))
    # response spans: one per group with response rows, in group order
    spans, g0, s = [], 0, 0
    for lp, g in zip(plens, gsz):
        pe = g0 + lp
        gend = pe + sum(rs[s:s + g])
        s += g
        if gend > pe:
            spans.append([pe, gend, g0, pe, pe, gend, 0, 0])
        g0 = gend
    assert st.n_tiles[5] == len(spans) and lists[5].tolist() == spans
    assert st.max_response_rows == max([sp[1] - sp[0] for sp in spans], default=0)
    for w, bm in [(2, 64), (3, 128)]:
        bt = lists[w]
        covered = torch.zeros(T, dtype=torch.int32)
        for k0, k1, q_lo, q_hi, g0, pe, _, _ in bt.tolist():
            assert 0 < k1 - k0 <= bm
            covered[k0:k1] += 1
            rows = torch.zeros(T, dtype=torch.bool)
            rows[q_lo:q_hi] = True
            assert not bool((mask[:, k0:k1] & ~rows[:, None]).any())
        assert torch.equal(covered, torch.ones(T, dtype=torch.int32))


def test_work_lists_are_heaviest_first():
    _, tab, st = api.pack_host([1000], [4], [100, 300, 50, 7])
    _, lists = unpack(tab, st)
    ft = lists[1].tolist()
    cost = [(q1 - q0) * ((p_end - g0) + (s_hi - s_lo)) for q0, q1, g0, p_end, s_lo, s_hi, _, _ in ft]
    assert cost == sorted(cost, reverse=True)


@pytest.mark.parametrize("plens,gsz,rs", [
    ([-1], [1], [3]), ([4], [-1], []), ([4], [2], [3, -2]), ([0], [1], [0]), ([], [], []),
])
def test_pack_rejects_bad_lengths(plens, gsz, rs):
    with pytest.raises(_lib.PgError) as e:
        api.pack_size(plens, gsz, rs)
    assert e.value.status == _lib.PG_ERR_INVALID_ARG


def test_attention_rejects_bad_arguments_on_host():
    _, tab, st = api.pack_host([8], [1], [4])
    L = _lib.lib()
    n = C.c_size_t()
    opts = _lib.PgOpts(0.0, 0.0, 0, 0)
    for hq, hkv, d in [(3, 2, 128), (4, 2, 96), (0, 1, 64)]:
        assert L.pg_workspace_size(C.byref(st), _lib.PG_BF16, hq, hkv, d, C.byref(opts), 0,
                                   C.byref(n)) == _lib.PG_ERR_INVALID_ARG
    assert L.pg_workspace_size(C.byref(st), _lib.PG_BF16, 4, 2, 128, C.byref(opts), 0,
                               C.byref(n)) == _lib.PG_OK
    # NULL and misaligned pointers are refused before anything is launched
    buf = torch.empty(4096, dtype=torch.uint8)
    p = C.c_void_p(buf.data_ptr())
    bad = C.c_void_p(buf.data_ptr() + 4)
    args = [C.byref(st), _lib.PG_BF16, 4, 2, 128]
    assert L.pg_grouped_attn_fwd(*args, None, p, p, p, p, C.byref(opts), p, 4096, None) \
        == _lib.PG_ERR_INVALID_ARG
    assert L.pg_grouped_attn_fwd(*args, p, bad, p, p, p, C.byref(opts), p, 4096, None) \
        == _lib.PG_ERR_INVALID_ARG
    assert b"16-byte" in L.pg_last_error_message()
    # the responses-only option is forward-only
    ro = _lib.PgOpts(0.0, 0.0, _lib.PG_FLAG_RESPONSES_ONLY, 0)
    assert L.pg_grouped_attn_bwd(*args, p, p, p, p, p, p, p, p, p, C.byref(ro), p, 4096, None) \
        == _lib.PG_ERR_INVALID_ARG
    assert b"forward-only" in L.pg_last_error_message()
    neg = _lib.PgOpts(-1.0, 0.0, 0, 0)
    assert L.pg_grouped_attn_fwd(*args, p, p, p, p, p, C.byref(neg), p, 4096, None) \
        == _lib.PG_ERR_INVALID_ARG


@pytest.mark.parametrize("B,Lp,G,R,rl", [
    (2, 5, 3, 4, [4, 0, 2, 1, 4, 3]),
    (1, 0, 2, 3, [1, 3]),
    (3, 7, 1, 0, [0, 0, 0]),
])
def test_padded_layout_is_full_slot_packing_plus_pad_rows(B, Lp, G, R, rl):
    # A padded batch is the packing with every response at max_response_len tokens; the layout
    # additionally lists exactly the slot tails beyond each response's length.
    pos, tab, st = api.pack_padded_host(B, Lp, G, R, rl)
    pos2, tab2, st2 = api.pack_host([Lp] * B, [G] * B, [R] * (B * G))
    assert torch.equal(pos, pos2) and st.total_tokens == st2.total_tokens == B * (Lp + G * R)
    assert tab.numpy().tobytes()[:st2.table_bytes] == tab2.numpy().tobytes()
    expect = []
    for b in range(B):
        for i in range(G):
            s0 = b * (Lp + G * R) + Lp + i * R
            expect += list(range(s0 + rl[b * G + i], s0 + R))
    assert st.n_pad_rows == len(expect)
    raw = tab.numpy().tobytes()[st.off_pad_rows: st.off_pad_rows + 4 * len(expect)]
    assert torch.frombuffer(bytearray(raw), dtype=torch.int32).tolist() == expect if expect else True


def test_padded_layout_rejects_bad_lengths():
    with pytest.raises(_lib.PgError):
        api.pack_padded_size(1, 4, 2, 3, [4, 1])
    with pytest.raises(_lib.PgError):
        api.pack_padded_size(1, 4, 2, 3, [-1, 1])


TREE_CASES = [
    ([-1, 0, 1, 1, 0, 4, 4, 4], [300, 70, 90, 130, 64, 1, 200, 65]),   # two turns, ragged
    ([-1, 0, 1, 2, 2, 0, -1, 6, 6], [129, 64, 300, 7, 70, 5, 80, 40, 0]),  # depth 4, two roots
    ([-1, 0, 0, 2, 2, 2], [0, 33, 100, 64, 1, 250]),                    # empty root
    ([-1, 0, 0, 0], [257, 31, 1, 200]),                                 # two-level
    ([-1, 0, 1, 2, 3, 4, 5, 6], [70, 3, 66, 1, 128, 9, 64, 300]),       # depth 8 chain
]


def tree_tables(parent, lens):
    pos, tab, st = api.pack_tree_host(parent, lens)
    raw = tab.numpy().tobytes()
    T = st.total_tokens
    tok = torch.frombuffer(bytearray(raw[st.off_tokens: st.off_tokens + 16 * T]),
                           dtype=torch.int32).view(T, 4)
    ivs = torch.frombuffer(bytearray(raw[st.off_intervals: st.off_intervals + 8 * st.n_intervals]),
                           dtype=torch.int32).view(-1, 2) if st.n_intervals else torch.zeros((0, 2))
    lists = []
    for w in range(5):
        n, o = st.n_tiles[w], st.off_tiles[w]
        lists.append(torch.frombuffer(bytearray(raw[o: o + 32 * n]), dtype=torch.int32).view(n, 8)
                     if n else torch.zeros((0, 8), dtype=torch.int32))
    return pos, tok, ivs, lists, st


@pytest.mark.parametrize("case", TREE_CASES)
def test_tree_tables_expand_to_the_tree_visibility(case):
    # The kernels' rules applied to every tile reproduce the oracle's visibility exactly.
    parent, lens = case
    pos, tok, ivs, lists, st = tree_tables(parent, lens)
    tl = orc.tree_layout(parent, lens)
    mask = orc.tree_visibility(tl)
    T = tl.total_tokens
    assert st.total_tokens == T and torch.equal(pos.to(torch.int64), tl.position_ids)
    assert st.pairs == int(mask.sum()) and st.num_groups == sum(p < 0 for p in parent)
    t_idx = torch.arange(T)
    for w, bm in [(0, 64), (1, 128), (4, 256)]:
        got = torch.zeros((T, T), dtype=torch.bool)
        covered = torch.zeros(T, dtype=torch.int32)
        for q0, q1, g0, p_end, s_lo, s_hi, a_off, a_cnt in lists[w].tolist():
            assert 0 < q1 - q0 <= bm and a_cnt <= 6
            covered[q0:q1] += 1
            causal = [(g0, p_end)] + [tuple(ivs[a_off + i].tolist()) for i in range(a_cnt)]
            for t in range(q0, q1):
                for lo, hi in causal:
                    got[t, lo:min(hi, t + 1)] = True
                own = int(tok[t, 2])
                got[t, max(s_lo, own):min(s_hi, t + 1)] = True
        assert torch.equal(covered, torch.ones(T, dtype=torch.int32))
        assert torch.equal(got, mask), bm
    for w, bm in [(2, 64), (3, 128)]:
        got = torch.zeros((T, T), dtype=torch.bool)
        for k0, k1, q_lo, q_hi, g0, pe, _, _ in lists[w].tolist():
            assert 0 < k1 - k0 <= bm
            own = tok[:, 2]
            for s in range(k0, k1):
                vis = (t_idx >= s) & (t_idx < q_hi) & ((s < pe) | (own <= s))
                got[:, s] |= vis
        assert torch.equal(got, mask), bm


def test_tree_layout_rejects_bad_trees():
    with pytest.raises(_lib.PgError) as e:
        api.pack_tree_size([-1, 0, -1, 1], [3, 2, 2, 1])     # node 3's parent is not on the path
    assert e.value.status == _lib.PG_ERR_INVALID_ARG
    with pytest.raises(_lib.PgError) as e:
        api.pack_tree_size([-1, 2, 0], [3, 2, 2])            # parent listed after the child
    assert e.value.status == _lib.PG_ERR_INVALID_ARG
    with pytest.raises(_lib.PgError) as e:
        api.pack_tree_size(list(range(-1, 8)), [4] * 9)      # depth 9
    assert e.value.status == _lib.PG_ERR_UNSUPPORTED


def test_keep_rotated_forward_needs_the_backward_workspace():
    _, tab, st = api.pack_host([300], [2], [40, 60])
    L = _lib.lib()
    n0, n1, nk = C.c_size_t(), C.c_size_t(), C.c_size_t()
    plain = _lib.PgOpts(0.0, 1e4, 0, 0)
    keep = _lib.PgOpts(0.0, 1e4, _lib.PG_FLAG_KEEP_ROTATED, 0)
    assert L.pg_workspace_size(C.byref(st), _lib.PG_BF16, 4, 2, 128, C.byref(plain), 0,
                               C.byref(n0)) == _lib.PG_OK
    assert L.pg_workspace_size(C.byref(st), _lib.PG_BF16, 4, 2, 128, C.byref(plain), 1,
                               C.byref(n1)) == _lib.PG_OK
    assert L.pg_workspace_size(C.byref(st), _lib.PG_BF16, 4, 2, 128, C.byref(keep), 0,
                               C.byref(nk)) == _lib.PG_OK
    assert n0.value < n1.value == nk.value


def test_responses_only_refuses_nested_layouts():
    # Scoring needs a two-level layout; a depth-3 tree is refused on the host, before any launch.
    _, tab, st = api.pack_tree_host([-1, 0, 1], [8, 4, 2])
    L = _lib.lib()
    buf = torch.empty(1 << 16, dtype=torch.uint8)
    p = C.c_void_p(buf.data_ptr())
    ro = _lib.PgOpts(0.0, 0.0, _lib.PG_FLAG_RESPONSES_ONLY, 0)
    assert L.pg_grouped_attn_fwd(C.byref(st), _lib.PG_BF16, 2, 1, 128, p, p, p, p, p, C.byref(ro),
                                 p, 1 << 16, None) == _lib.PG_ERR_UNSUPPORTED


def test_tree_packing_matches_hand_fixture():
    import json
    fx = json.load(open(os.path.join(ROOT, "tests", "golden", "pack_tree_small.json")))
    pos, tok, ivs, lists, st = tree_tables(fx["parent"], fx["seg_lens"])
    assert st.total_tokens == fx["total_tokens"] and st.pairs == fx["grouped_pairs"]
    assert pos.tolist() == fx["position_ids"]
    assert st.max_depth == 3


def test_pre_rotated_workspace_and_argument_checks():
    # With q and k arriving rotated the backward's workspace holds no rotated copies of them, only
    # the cos/sin table; the flag needs RoPE; the table call and the RoPE GEMM check their
    # arguments on the host (nothing here reaches a launch).
    _, tab, st = api.pack_host([300], [2], [40, 60])
    T, Hq, Hkv, d = st.total_tokens, 4, 2, 128
    L = _lib.lib()
    pre, keep = _lib.PG_FLAG_PRE_ROTATED, _lib.PG_FLAG_KEEP_ROTATED

    def size(flags, theta, phase):
        n = C.c_size_t()
        rc = L.pg_workspace_size(C.byref(st), _lib.PG_BF16, Hq, Hkv, d,
                                 C.byref(_lib.PgOpts(0.0, theta, flags, 0)), phase, C.byref(n))
        return rc, n.value

    def al(b):
        return (b + 255) // 256 * 256

    rc0, plain1 = size(0, 1e4, 1)
    rc1, pre1 = size(pre, 1e4, 1)
    assert rc0 == rc1 == _lib.PG_OK
    assert plain1 - pre1 == al(T * Hq * d * 2) + al(T * Hkv * d * 2)
    assert size(pre, 1e4, 0) == (_lib.PG_OK, 0)
    assert size(pre | keep, 1e4, 0) == (_lib.PG_OK, pre1)
    assert size(pre, 0.0, 1)[0] == _lib.PG_ERR_INVALID_ARG

    buf = torch.empty(1 << 16, dtype=torch.uint8)
    p = C.c_void_p(buf.data_ptr())
    out = C.c_void_p()

    def table(flags, theta, nbytes):
        return L.pg_rope_table(C.byref(st), _lib.PG_BF16, Hq, Hkv, d,
                               C.byref(_lib.PgOpts(0.0, theta, flags, 0)), p, nbytes,
                               C.byref(out), None)

    assert table(0, 1e4, pre1) == _lib.PG_ERR_INVALID_ARG          # flag missing
    assert table(pre, 0.0, pre1) == _lib.PG_ERR_INVALID_ARG        # no RoPE
    assert table(pre, 1e4, pre1 - 1) == _lib.PG_ERR_INVALID_ARG    # workspace too small

    def gemm(M, N, K, ldc, hd, tab_ptr, rows):
        return L.pg_gemm_bf16_rope(M, N, K, p, K, p, K, p, ldc, hd, tab_ptr, rows, None)

    assert gemm(256, 384, 64, 384, 96, p, 256) == _lib.PG_ERR_INVALID_ARG     # head_dim
    assert gemm(256, 320, 64, 320, 128, p, 256) == _lib.PG_ERR_INVALID_ARG    # N % head_dim
    assert gemm(256, 384, 64, 384, 128, p, 255) == _lib.PG_ERR_INVALID_ARG    # table too short
    assert gemm(256, 384, 64, 384, 128, None, 256) == _lib.PG_ERR_INVALID_ARG  # no table
    assert gemm(256, 384, 64, 388, 128, p, 256) == _lib.PG_ERR_INVALID_ARG    # ldc % 8
    assert gemm(256, 384, 64, 384, 96, p, 256) == _lib.PG_ERR_INVALID_ARG
    assert b"head_dim" in L.pg_last_error_message()
