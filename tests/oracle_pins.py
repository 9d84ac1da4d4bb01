"""Pins for the fp64 oracle: facts from the pages and from mathematics.

Every function ``pin_*`` takes an ``oracle.oracle.Oracle`` and raises
AssertionError when the oracle disagrees with the fact it checks.  They run
against the real oracle (test_oracle_pins.py) and against deliberately broken
copies of it (test_oracle_mutants.py), where at least one pin must fail.

The inputs are tiny and built here with numpy only; no pin compares the
oracle with a retyped copy of its own formula.
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers --

def to_bf16_bits(x) -> np.ndarray:
    """float -> bf16 bit patterns, round-to-nearest-even (finite inputs)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def from_bf16_bits(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def read_table(name: str):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows


def ints(s: str):
    return [int(v) for v in s.split()]


class Case:
    """A tiny batch built from *logical* per-request contexts.

    The test places each request's logical K/V rows into randomly chosen
    physical blocks itself; the expected attention is then computed from the
    logical rows alone, with no paging involved.
    """

    def __init__(self, rng, *, hq, hkv, d, q_lens, seq_lens, num_blocks=None, bs=16,
                 kv=None, qv=None, poison=3.0e4):
        self.hq, self.hkv, self.d, self.bs = hq, hkv, d, bs
        self.q_lens = np.asarray(q_lens, dtype=np.int64)
        self.seq_lens = np.asarray(seq_lens, dtype=np.int64)
        self.num_computed = self.seq_lens - self.q_lens
        R = len(self.seq_lens)
        self.qsl = np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)
        T = int(self.qsl[-1])
        nblk = (self.seq_lens + bs - 1) // bs
        self.num_blocks = int(num_blocks or (nblk.sum() + 3))
        maxb = int(max(1, nblk.max()))
        perm = rng.permutation(self.num_blocks)
        self.block_table = np.full((R, maxb), perm[-1], dtype=np.int32)  # padding -> last id
        c = 0
        for r in range(R):
            self.block_table[r, :nblk[r]] = perm[c:c + nblk[r]]
            c += nblk[r]
        # logical contexts, exactly representable in bf16
        if kv is None:
            self.k_log = [from_bf16_bits(to_bf16_bits(rng.standard_normal((L, hkv, d)))) for L in self.seq_lens]
            self.v_log = [from_bf16_bits(to_bf16_bits(rng.standard_normal((L, hkv, d)))) for L in self.seq_lens]
        else:
            self.k_log, self.v_log = kv
        self.q = from_bf16_bits(to_bf16_bits(rng.standard_normal((T, hq, d)))) if qv is None else qv
        # physical caches: poison everywhere, then logical rows into place
        pois = np.where(np.arange(self.num_blocks * bs * hkv * d) % 2 == 0, poison, -poison)
        self.kc = to_bf16_bits(pois).reshape(self.num_blocks, bs, hkv, d)
        self.vc = to_bf16_bits(-pois).reshape(self.num_blocks, bs, hkv, d)
        for r in range(R):
            for j in range(int(self.seq_lens[r])):
                blk = self.block_table[r, j // bs]
                self.kc[blk, j % bs] = to_bf16_bits(self.k_log[r][j])
                self.vc[blk, j % bs] = to_bf16_bits(self.v_log[r][j])
        self.scale = 1.0 / math.sqrt(d)

    def run(self, orc, rows=None, **over):
        kw = dict(query_start_loc=self.qsl, seq_lens=self.seq_lens.astype(np.int32),
                  num_computed=self.num_computed.astype(np.int32), block_table=self.block_table,
                  q=to_bf16_bits(self.q), key_cache=self.kc, value_cache=self.vc,
                  softmax_scale=self.scale, rows=rows)
        kw.update(over)
        return orc.attention(**kw)

    def dense_expected(self):
        """Matrix-form attention from the logical contexts (numpy, fp64)."""
        T = int(self.qsl[-1])
        out = np.zeros((T, self.hq, self.d))
        g = self.hq // self.hkv
        for r in range(len(self.seq_lens)):
            a, b = int(self.qsl[r]), int(self.qsl[r + 1])
            if a == b:
                continue
            L = int(self.seq_lens[r])
            c = int(self.num_computed[r])
            pos = c + np.arange(b - a)
            visible = np.arange(L)[None, :] <= pos[:, None]            # [q, L]
            for h in range(self.hq):
                K = self.k_log[r][:, h // g, :]                          # [L, d]
                V = self.v_log[r][:, h // g, :]
                S = self.scale * (self.q[a:b, h, :] @ K.T)               # [q, L]
                S = np.where(visible, S, -np.inf)
                P = np.exp(S - S.max(axis=1, keepdims=True))
                P /= P.sum(axis=1, keepdims=True)
                out[a:b, h, :] = P @ V
        return out


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------- pins --

def pin_slot_examples(orc):
    """Worked slot examples of §6.3 and §10.1 (golden/slot_examples.txt)."""
    for name, bs, nc, ql, row, slots in read_table("slot_examples.txt"):
        qsl = np.array([0, int(ql)], dtype=np.int32)
        table = np.array([ints(row)], dtype=np.int32)
        got = orc.slot_mapping(qsl, np.array([int(nc)], dtype=np.int32), table, int(bs))
        assert got.tolist() == ints(slots), (name, got.tolist(), slots)


def pin_mixed_batch_metadata(orc):
    """The R0/R1/R2 example: lengths consistent with query_start_loc are
    accepted; R1's first new token lands at position 512 (its prefix hit)."""
    for name, sched, comp, qsl, seq in read_table("mixed_batch_example.txt"):
        sched, comp, qsl, seq = ints(sched), ints(comp), ints(qsl), ints(seq)
        assert np.concatenate([[0], np.cumsum(sched)]).tolist() == qsl, name
        R = len(sched)
        maxb = max(1, max((s + 15) // 16 for s in seq))
        table = np.arange(R * maxb, dtype=np.int32).reshape(R, maxb)
        slots = orc.slot_mapping(np.array(qsl, np.int32), np.array(comp, np.int32), table, 16)
        for r in range(R):
            assert slots[qsl[r]] == table[r, comp[r] // 16] * 16 + comp[r] % 16, name
        # attention accepts the metadata (tiny heads) ...
        rng = _rng(5)
        case = Case(rng, hq=2, hkv=1, d=64, q_lens=sched, seq_lens=seq)
        case.run(orc, rows=[0, qsl[-1] - 1])
        # ... and rejects an inconsistent num_computed
        bad = case.num_computed.copy()
        bad[-1] += 1
        try:
            case.run(orc, rows=[0], num_computed=bad.astype(np.int32))
        except RuntimeError:
            pass
        else:
            raise AssertionError("inconsistent num_computed accepted")


def pin_write_bit_copy(orc):
    """reshape_and_cache scatter: slot s receives token t's full row, bit for
    bit; negative slots write nothing; other slots keep their contents."""
    rng = _rng(1)
    nb, bs, hkv, d, T = 6, 16, 2, 64, 20
    kc = rng.integers(0, 65536, size=(nb, bs, hkv, d), dtype=np.uint16)
    vc = rng.integers(0, 65536, size=(nb, bs, hkv, d), dtype=np.uint16)
    key = rng.integers(0, 65536, size=(T, hkv, d), dtype=np.uint16)
    val = rng.integers(0, 65536, size=(T, hkv, d), dtype=np.uint16)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[[3, 11]] = -1
    ek, ev = kc.copy(), vc.copy()
    for t in range(T):
        if slots[t] >= 0:
            ek[slots[t] // bs, slots[t] % bs] = key[t]
            ev[slots[t] // bs, slots[t] % bs] = val[t]
    gk, gv = kc.copy(), vc.copy()
    assert orc.write_kv(key, val, slots, gk, gv) == 0
    assert np.array_equal(gk, ek) and np.array_equal(gv, ev)


def pin_single_visible_key(orc):
    """A request of length 1: the only visible key has weight 1, out = v_0."""
    rng = _rng(2)
    case = Case(rng, hq=4, hkv=2, d=64, q_lens=[1], seq_lens=[1])
    out = case.run(orc)
    g = 2
    for h in range(4):
        assert np.array_equal(out[0, h], case.v_log[0][0, h // g]), h


def pin_zero_query(orc):
    """q = 0 gives equal weights: out = mean of the visible value rows."""
    rng = _rng(3)
    T = 7
    case = Case(rng, hq=2, hkv=1, d=64, q_lens=[T], seq_lens=[T + 9], qv=np.zeros((T, 2, 64)))
    out = case.run(orc)
    for i in range(T):
        vis = 9 + i + 1
        mean = case.v_log[0][:vis, 0].mean(axis=0)
        assert np.allclose(out[i, 0], mean, rtol=0, atol=1e-12), i


def pin_identical_keys(orc):
    """All keys equal: every score is the same, out = mean of V."""
    rng = _rng(4)
    L = 37
    k_row = from_bf16_bits(to_bf16_bits(rng.standard_normal((1, 1, 64))))
    k = np.repeat(k_row, L, axis=0)
    v = from_bf16_bits(to_bf16_bits(rng.standard_normal((L, 1, 64))))
    case = Case(rng, hq=1, hkv=1, d=64, q_lens=[1], seq_lens=[L], kv=([k], [v]))
    out = case.run(orc)
    assert np.allclose(out[0, 0], v[:, 0].mean(axis=0), rtol=0, atol=1e-12)


def pin_two_keys_closed_form(orc):
    """Two keys: out = v0 + sigmoid(s1 - s0) (v1 - v0) with s = <q,k>/sqrt(D).

    q = e_0, k0 = 0, k1 = 4 e_0 + 4 e_1, D = 64: s0 = 0, s1 = 4/8 = 0.5.
    """
    d = 64
    k = np.zeros((2, 1, d)); k[1, 0, 0] = 4.0; k[1, 0, 1] = 4.0
    v = np.zeros((2, 1, d)); v[0, 0, :] = 1.0; v[1, 0, :] = -2.0
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 1.0
    case = Case(_rng(6), hq=1, hkv=1, d=d, q_lens=[1], seq_lens=[2], kv=([k], [v]), qv=q)
    out = case.run(orc)
    w1 = 1.0 / (1.0 + math.exp(-0.5))
    expect = 1.0 + w1 * (-3.0)
    assert np.allclose(out[0, 0], expect, rtol=0, atol=1e-14), (out[0, 0, 0], expect)


def pin_dominant_key(orc):
    """One score far above the rest: out = that key's value row."""
    d, L, hot = 64, 30, 17
    rng = _rng(7)
    k = from_bf16_bits(to_bf16_bits(rng.standard_normal((L, 1, d)) * 0.01))
    k[hot, 0, :] = 16.0
    v = from_bf16_bits(to_bf16_bits(rng.standard_normal((L, 1, d))))
    q = np.full((1, 1, d), 16.0)
    case = Case(rng, hq=1, hkv=1, d=d, q_lens=[1], seq_lens=[L], kv=([k], [v]), qv=q)
    out = case.run(orc)
    assert np.allclose(out[0, 0], v[hot, 0], rtol=0, atol=1e-12)


def pin_gqa_mapping(orc):
    """Query head h reads kv head h // (Hq/Hkv): contiguous head groups."""
    hq, hkv, d, L = 8, 2, 64, 20
    rng = _rng(8)
    k = from_bf16_bits(to_bf16_bits(rng.standard_normal((L, hkv, d))))
    v = np.zeros((L, hkv, d)); v[:, 0, :] = -3.0; v[:, 1, :] = 7.0
    case = Case(rng, hq=hq, hkv=hkv, d=d, q_lens=[3], seq_lens=[L], kv=([k], [v]))
    out = case.run(orc)
    for h in range(hq):
        assert np.allclose(out[:, h], -3.0 if h < 4 else 7.0, atol=1e-12), h


def pin_causal_visibility(orc):
    """Query i of a chunk over c cached tokens sees keys 0..c+i: changing a
    later key leaves it alone, changing key c+i (its own) changes it."""
    rng = _rng(9)
    c, n = 21, 6
    base = Case(rng, hq=2, hkv=1, d=64, q_lens=[n], seq_lens=[c + n])
    out0 = base.run(orc)
    for i in range(n - 1):
        k2 = base.k_log[0].copy(); v2 = base.v_log[0].copy()
        k2[c + i + 1:] = -k2[c + i + 1:] + 1.0
        v2[c + i + 1:] = 5.0
        alt = Case(_rng(99), hq=2, hkv=1, d=64, q_lens=[n], seq_lens=[c + n],
                   kv=([k2], [v2]), qv=base.q)
        out1 = alt.run(orc)
        assert np.array_equal(out0[:i + 1], out1[:i + 1]), i
        k3 = base.k_log[0].copy(); v3 = base.v_log[0].copy()
        v3[c + i] = 5.0
        alt2 = Case(_rng(98), hq=2, hkv=1, d=64, q_lens=[n], seq_lens=[c + n],
                    kv=([k3], [v3]), qv=base.q)
        out2 = alt2.run(orc)
        assert not np.allclose(out0[i], out2[i]), i


def pin_decode_equals_last_prefill_row(orc):
    """A decode step over L-1 cached tokens equals the last row of a prefill
    of all L tokens (§10.1 prefill, §10.2 decode)."""
    rng = _rng(10)
    L = 45
    pre = Case(rng, hq=4, hkv=2, d=64, q_lens=[L], seq_lens=[L])
    out_p = pre.run(orc)
    dec = Case(_rng(11), hq=4, hkv=2, d=64, q_lens=[1], seq_lens=[L],
               kv=(pre.k_log, pre.v_log), qv=pre.q[L - 1:L])
    out_d = dec.run(orc)
    assert np.array_equal(out_p[L - 1], out_d[0])


def pin_prefix_hit_equals_recompute(orc):
    """A request whose first 32 tokens hit the prefix cache (num_computed 32)
    gives the same rows as recomputing the whole prompt (§10.3)."""
    rng = _rng(12)
    L, hit = 50, 32
    full = Case(rng, hq=2, hkv=1, d=64, q_lens=[L], seq_lens=[L])
    out_f = full.run(orc)
    part = Case(_rng(13), hq=2, hkv=1, d=64, q_lens=[L - hit], seq_lens=[L],
                kv=(full.k_log, full.v_log), qv=full.q[hit:])
    out_h = part.run(orc)
    assert np.array_equal(out_f[hit:], out_h)


def pin_block_permutation(orc):
    """Physical placement only changes addressing: two different random
    placements of the same logical contexts give identical outputs."""
    rng = _rng(14)
    a = Case(rng, hq=4, hkv=2, d=64, q_lens=[1, 9, 1], seq_lens=[40, 9, 17])
    b = Case(_rng(15), hq=4, hkv=2, d=64, q_lens=[1, 9, 1], seq_lens=[40, 9, 17],
             kv=(a.k_log, a.v_log), qv=a.q, num_blocks=a.num_blocks + 5)
    assert not np.array_equal(a.block_table[:, :1], b.block_table[:, :1])
    assert np.array_equal(a.run(orc), b.run(orc))


def pin_partition_merge(orc):
    """Splitting the keys into partitions and merging (m, l, o) gives the
    unsplit result (page and partition boundaries do not change it)."""
    rng = _rng(16)
    L = 70
    case = Case(rng, hq=2, hkv=1, d=64, q_lens=[1], seq_lens=[L])
    kw = dict(query_start_loc=case.qsl, seq_lens=case.seq_lens.astype(np.int32),
              num_computed=case.num_computed.astype(np.int32), block_table=case.block_table,
              q=to_bf16_bits(case.q), key_cache=case.kc, value_cache=case.vc,
              softmax_scale=case.scale)
    whole = orc.attention_range(**kw)
    for cuts in ([0, 16, 70], [0, 5, 33, 64, 70], [0, 69, 70], [0, 1, 2, 3, 70]):
        parts = [orc.attention_range(**kw, key_begin=a, key_end=b) for a, b in zip(cuts[:-1], cuts[1:])]
        for h in range(2):
            o, m, l = orc.merge([p.m[0, h] for p in parts], [p.l[0, h] for p in parts],
                                np.stack([p.out[0, h] for p in parts]))
            assert np.allclose(o, whole.out[0, h], rtol=0, atol=1e-12), cuts
            assert math.isclose(m, whole.m[0, h], rel_tol=0, abs_tol=1e-12)
            assert math.isclose(l, whole.l[0, h], rel_tol=1e-12)
    # the partial of one range is its own softmax: m is the largest score
    p = orc.attention_range(**kw, key_begin=10, key_end=20)
    k = case.k_log[0][10:20, 0]
    s = case.scale * (k @ case.q[0, 0])
    assert math.isclose(p.m[0, 0], s.max(), abs_tol=1e-12)
    assert math.isclose(p.l[0, 0], np.exp(s - s.max()).sum(), rel_tol=1e-12)


def pin_dense_bruteforce(orc):
    """Random tiny mixed batches against the dense masked-matrix form."""
    for seed, hq, hkv, d in ((17, 4, 2, 64), (18, 8, 2, 128), (19, 4, 4, 64)):
        rng = _rng(seed)
        case = Case(rng, hq=hq, hkv=hkv, d=d, q_lens=[1, 7, 0, 1, 19],
                    seq_lens=[23, 7, 5, 1, 40])
        got = case.run(orc)
        want = case.dense_expected()
        assert np.allclose(got, want, rtol=0, atol=1e-12), seed


def pin_common_prefix_precondition(orc):
    """num_common_prefix_blocks: the shared blocks must be identical across
    requests with queries and fully computed by each of them."""
    table = np.array([[5, 6, 7, 8], [5, 6, 9, 10], [5, 11, 12, 13]], dtype=np.int32)
    qsl = np.array([0, 1, 2, 3], dtype=np.int32)
    nc = np.array([40, 40, 40], dtype=np.int32)
    assert orc.check_common_prefix(qsl, nc, table, 16, 0) == 0
    assert orc.check_common_prefix(qsl, nc, table, 16, 1) == 0
    assert orc.check_common_prefix(qsl, nc, table, 16, 2) != 0      # row 2 differs
    qsl2 = np.array([0, 1, 2, 2], dtype=np.int32)                   # row 2 idle
    assert orc.check_common_prefix(qsl2, nc, table, 16, 2) == 0
    table2 = np.array([[5, 6, 7, 8], [5, 6, 9, 10], [5, 6, 12, 13]], dtype=np.int32)
    assert orc.check_common_prefix(qsl, nc, table2, 16, 2) == 0
    nc2 = np.array([40, 31, 40], dtype=np.int32)                    # 2*16 > 31
    assert orc.check_common_prefix(qsl, nc2, table2, 16, 2) != 0
    assert orc.check_common_prefix(qsl, nc2, table2, 16, 1) == 0    # 16 <= 31


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


def run_all(orc):
    """Run every pin; return the names of those that failed."""
    failed = []
    for pin in PINS:
        try:
            pin(orc)
        except Exception:  # noqa: BLE001 -- any failure counts
            failed.append(pin.__name__)
    return failed


# ------------------------------------------------------------ FP8 (E4M3) --

def pin_e4m3_codes(orc):
    """Code <-> value pairs fixed by the E4M3 definition (golden/e4m3_codes.txt)."""
    for value, code in read_table("e4m3_codes.txt"):
        v, c = float(value), int(code, 16)
        assert orc.e4m3_encode(v) == c, (value, hex(orc.e4m3_encode(v)))
        got = orc.e4m3_value(c)
        assert got == v and math.copysign(1.0, got) == math.copysign(1.0, v), (code, got)


def pin_e4m3_round_trip_and_order(orc):
    """Every finite code survives decode -> encode; magnitudes grow with the
    code; the sign bit mirrors the value; 0x7F / 0xFF are NaN."""
    prev = -1.0
    for c in range(0x7F):
        v = orc.e4m3_value(c)
        assert orc.e4m3_encode(v) == c, hex(c)
        assert orc.e4m3_encode(-v) == (c | 0x80), hex(c)
        assert v > prev or (c == 0 and v == 0.0), hex(c)
        prev = v
    assert math.isnan(orc.e4m3_value(0x7F)) and math.isnan(orc.e4m3_value(0xFF))


def pin_e4m3_rounding(orc):
    """Nearest value, ties to the even mantissa, saturation at 448."""
    assert orc.e4m3_encode(1.0625) == 0x38          # halfway 1.0 / 1.125 -> even (1.0)
    assert orc.e4m3_encode(1.1875) == 0x3A          # halfway 1.125 / 1.25 -> even (1.25)
    assert orc.e4m3_encode(1.06) == 0x38 and orc.e4m3_encode(1.07) == 0x39   # either side of 1.0625
    assert orc.e4m3_encode(1.5 * 2 ** -9) == 0x02   # subnormal tie -> even
    assert orc.e4m3_encode(2 ** -11) == 0x00        # below half the smallest subnormal
    assert orc.e4m3_encode(0.99 * 2 ** -6) == 0x08  # rounds up into the normal range
    for big in (449.0, 463.9, 464.0, 500.0, 1e6, float("inf")):
        assert orc.e4m3_encode(big) == 0x7E and orc.e4m3_encode(-big) == 0xFE, big
    assert orc.e4m3_encode(float("nan")) == 0x7F


def pin_fp8_write_scales(orc):
    """The FP8 write stores the code of x / scale, K and V with their own scale."""
    nb, bs, hkv, d = 2, 16, 1, 64
    kc = np.zeros((nb, bs, hkv, d), np.uint8)
    vc = np.zeros((nb, bs, hkv, d), np.uint8)
    key = to_bf16_bits(np.full((3, hkv, d), 2.0))
    val = to_bf16_bits(np.full((3, hkv, d), -3.0))
    slots = np.array([5, -1, 20], np.int64)
    assert orc.write_kv_fp8(key, val, slots, kc, vc, 0.5, 2.0) == 0
    flat_k, flat_v = kc.reshape(-1, d), vc.reshape(-1, d)
    assert np.all(flat_k[5] == 0x48) and np.all(flat_k[20] == 0x48)      # 2 / 0.5 = 4
    assert np.all(flat_v[5] == 0xBC) and np.all(flat_v[20] == 0xBC)      # -3 / 2 = -1.5
    untouched = [i for i in range(nb * bs) if i not in (5, 20)]
    assert not flat_k[untouched].any() and not flat_v[untouched].any()


def _fp8_case(seed):
    """Tiny FP8 batch and a bf16 batch holding exactly its dequantised values
    (a power-of-two scale keeps every code_value * scale exact in bf16)."""
    rng = _rng(seed)
    case = Case(rng, hq=4, hkv=2, d=64, q_lens=[1, 9, 1], seq_lens=[37, 9, 20])
    codes_k = rng.integers(0, 256, size=case.kc.shape).astype(np.uint8)
    codes_v = rng.integers(0, 256, size=case.vc.shape).astype(np.uint8)
    for codes in (codes_k, codes_v):      # no NaN codes
        codes[(codes & 0x7F) == 0x7F] = 0x3A
    return case, codes_k, codes_v


def pin_fp8_attention_is_dequantised_attention(orc):
    """Attention over FP8 caches equals attention over the dequantised values."""
    case, ck, cv = _fp8_case(30)
    ks, vs = 0.25, 0.5
    vals_k = np.vectorize(orc.e4m3_value)(ck) * ks
    vals_v = np.vectorize(orc.e4m3_value)(cv) * vs
    kw = dict(query_start_loc=case.qsl, seq_lens=case.seq_lens.astype(np.int32),
              num_computed=case.num_computed.astype(np.int32), block_table=case.block_table,
              q=to_bf16_bits(case.q), softmax_scale=case.scale)
    got = orc.attention_fp8(key_cache=ck, value_cache=cv, k_scale=ks, v_scale=vs, **kw)
    want = orc.attention(key_cache=to_bf16_bits(vals_k), value_cache=to_bf16_bits(vals_v), **kw)
    assert np.allclose(got, want, rtol=0, atol=1e-12)


def pin_fp8_scale_roles(orc):
    """k_scale acts as a softmax temperature, v_scale multiplies the output."""
    case, ck, cv = _fp8_case(31)
    kw = dict(query_start_loc=case.qsl, seq_lens=case.seq_lens.astype(np.int32),
              num_computed=case.num_computed.astype(np.int32), block_table=case.block_table,
              q=to_bf16_bits(case.q), key_cache=ck, value_cache=cv)
    a = orc.attention_fp8(softmax_scale=case.scale, k_scale=0.02, v_scale=1.0, **kw)
    b = orc.attention_fp8(softmax_scale=case.scale * 2, k_scale=0.01, v_scale=1.0, **kw)
    c = orc.attention_fp8(softmax_scale=case.scale, k_scale=0.02, v_scale=3.0, **kw)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)
    assert np.allclose(c, 3.0 * a, rtol=1e-12, atol=1e-12)
    d = orc.attention_fp8(softmax_scale=case.scale, k_scale=0.04, v_scale=1.0, **kw)
    assert not np.allclose(a, d)


def pin_zero_blocks(orc):
    """new_block_ids_to_zero ("vLLM 推理流程分析" §4, §5.1.1): every byte of
    the K and V entries of each listed block becomes 0, nothing else changes,
    negative ids are skipped, an id past the cache is reported and skipped;
    the same holds for one-byte (E4M3) caches."""
    rng = _rng(40)
    for dtype, hi in ((np.uint16, 65536), (np.uint8, 256)):
        nb, bs, hkv, d = 7, 16, 2, 64
        kc = rng.integers(1, hi, size=(nb, bs, hkv, d), dtype=dtype)   # no zero byte pattern to hide in
        vc = rng.integers(1, hi, size=(nb, bs, hkv, d), dtype=dtype)
        gk, gv = kc.copy(), vc.copy()
        assert orc.zero_blocks(np.array([5, -1, 2]), gk, gv) == 0
        for b in range(nb):
            if b in (2, 5):
                assert not gk[b].any() and not gv[b].any(), b
            else:
                assert np.array_equal(gk[b], kc[b]) and np.array_equal(gv[b], vc[b]), b
        # idempotent and independent of the order of the ids
        hk, hv = kc.copy(), vc.copy()
        assert orc.zero_blocks(np.array([2, 5, 2]), hk, hv) == 0
        assert np.array_equal(hk, gk) and np.array_equal(hv, gv)
        # an id past the cache: status 2, the valid ids are still zeroed
        ik, iv = kc.copy(), vc.copy()
        assert orc.zero_blocks(np.array([nb, 0]), ik, iv) == 2
        assert not ik[0].any() and np.array_equal(ik[1:], kc[1:]) and np.array_equal(iv[1:], vc[1:])
    # a zeroed element reads as +0 in both element types
    assert orc.bf16_value(0) == 0.0 and math.copysign(1.0, orc.bf16_value(0)) == 1.0
    assert orc.e4m3_value(0) == 0.0 and math.copysign(1.0, orc.e4m3_value(0)) == 1.0


def pin_zeroed_tail_is_never_read(orc):
    """The reason for zeroing (§5.1.1): slots of a new block not yet written
    must not reach the result.  A decode whose last block was zeroed and then
    written in part gives the dense result, and the same result when the
    unwritten slots hold +inf / NaN instead of zeros."""
    case = Case(_rng(41), hq=4, hkv=2, d=64, q_lens=[1], seq_lens=[21], num_blocks=4)
    blk = int(case.block_table[0, 1])
    a_k, a_v = case.kc.copy(), case.vc.copy()
    assert orc.zero_blocks(np.array([blk]), a_k, a_v) == 0
    a_k[blk, :5], a_v[blk, :5] = case.kc[blk, :5], case.vc[blk, :5]      # keys 16..20 written
    b_k, b_v = a_k.copy(), a_v.copy()
    b_k[blk, 5:], b_v[blk, 5:] = 0x7F80, 0x7FC0                           # +inf / NaN, never written
    out_a = case.run(orc, key_cache=a_k, value_cache=a_v)
    out_b = case.run(orc, key_cache=b_k, value_cache=b_v)
    assert np.array_equal(out_a, out_b)
    assert np.max(np.abs(out_a - case.dense_expected())) < 1e-12


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
