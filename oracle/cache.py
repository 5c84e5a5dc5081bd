"""Region model of one KV head of one layer of one sequence (test infrastructure).

SJ-KVaRN §2.1 "The life of a token": a token passes through up to four regions — a
128-token 16-bit sink, a rotated 6.125-bit staging ring (tq6_0), the newest tokens read
at near-full precision, and compact body records made by a batched seal of every full
128-token group older than the newest ``keep`` tokens. KV Cache Precision Tail §2: the
newest N rows are read from an exact BF16/F16 store, older rows from quantized records,
under one softmax. Reading (the pages use "tail" for both): the tq6_0 ring holds every
unsealed position past the sink, and a separate exact store keeps a verbatim copy of the
newest T positions; configurations without a tq6_0 ring keep an F16/BF16 journal, which
is itself the exact store.

The model follows the format specification step by step: ``append`` writes one or more
positions, ``seal`` turns full groups into records, ``regions`` returns the dequantized
content of every region for the attention oracle, ``record_bytes`` the stored bytes of a
body record for byte-exact comparison.
"""

from dataclasses import dataclass

import numpy as np

from . import codecs, kvarn
from .fp import bf16_bits_from_f32, bf16_bits_to_f32, f16_bits
from .rotation import rotate, NONE, HAD256, TBQ128

SINK = 128
GROUP = 128


def rotation_of(fmt):
    if fmt in ("tbq4", "turbo3", "tq5_0"):
        return TBQ128
    if fmt.startswith("kvarn"):
        return HAD256
    if fmt in ("q8_0", "q4_0", "q5_0", "q6_0", "q4_1", "q5_1"):
        return NONE
    raise ValueError(fmt)


@dataclass(frozen=True)
class HeadConfig:
    head_dim: int
    k_body: str            # tbq4 | turbo3 | tq5_0 | q8_0 | q4_0 | q5_0 | q6_0 | q4_1 | q5_1 | kvarn2..kvarn8
    v_body: str
    journal: str           # tq6_0 | f16 | bf16
    tail_fmt: str          # f16 | bf16 (exact tail store; with an exact journal, its format)
    tail: int              # T
    ring: int              # R, journal capacity (positions)
    kvarn_balance: str = "final16"   # KVarN balancing: "final16" or "best8" (kvarn.BALANCE_MODES)

    @property
    def rot(self):
        r = rotation_of(self.k_body)
        assert rotation_of(self.v_body) == r, "K and V bodies must share a rotation"
        return r


def _store_exact(x_f16, fmt):
    """fp16 input -> stored 16-bit pattern in the exact format (verbatim or bf16 RNE)."""
    if fmt == "f16":
        return f16_bits(x_f16)
    return bf16_bits_from_f32(np.asarray(x_f16, dtype=np.float16).astype(np.float32))


def _load_exact(bits, fmt):
    if fmt == "f16":
        return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)
    return bf16_bits_to_f32(bits)


def encode_body(X, fmt, kvarn_balance="final16"):
    """Rows X [128, D] fp32 in the body's domain -> unpacked record fields."""
    if fmt == "tbq4":
        n16, idx = codecs.tbq4_encode(X)
        return {"scale": n16, "code": idx.reshape(X.shape)}
    if fmt == "q8_0":
        d, q = codecs.q8_encode(X)
        return {"scale": d, "code": q.reshape(X.shape)}
    if fmt == "q4_0":
        d, c = codecs.q4_encode(X)
        return {"scale": d, "code": c.reshape(X.shape)}
    if fmt == "turbo3":
        n16, idx = codecs.turbo3_encode(X)
        return {"scale": n16, "code": idx.reshape(X.shape)}
    if fmt == "tq5_0":
        d, c = codecs.tq5_encode(X)
        return {"scale": d, "code": c.reshape(X.shape)}
    if fmt in QSYM:
        d, c = codecs.qsym_encode(X, QSYM[fmt])
        return {"scale": d, "code": c.reshape(X.shape)}
    if fmt in QMIN:
        d, m, c = codecs.qmin_encode(X, QMIN[fmt])
        return {"scale": d, "min": m, "code": c.reshape(X.shape)}
    if fmt.startswith("kvarn"):
        bits = int(fmt[5:])
        D = X.shape[-1]
        tiles = X.reshape(128, D // 256, 256).transpose(1, 0, 2)   # [half, 128, 256]
        code, S, Z, C = kvarn.encode(tiles, bits, kvarn_balance)
        return {"code": code, "S": S, "Z": Z, "C": C, "bits": bits}
    raise ValueError(fmt)


# 32-value block formats beyond Q8_0 / Q4_0: symmetric levels L, or min-offset levels Q
QSYM = {"q5_0": 15, "q6_0": 31}
QMIN = {"q4_1": 15, "q5_1": 31}
CODE_BITS = {"q5_0": 5, "q6_0": 6, "q4_1": 4, "q5_1": 5}


def decode_body(rec, fmt):
    """Unpacked record -> dequantized rows [128, D] fp32 (rotated domain)."""
    if fmt == "tbq4":
        D = rec["code"].shape[-1]
        return codecs.tbq4_decode(rec["scale"], rec["code"].reshape(128, D // 128, 128))
    if fmt == "q8_0":
        D = rec["code"].shape[-1]
        return codecs.q8_decode(rec["scale"], rec["code"].reshape(128, D // 32, 32))
    if fmt == "q4_0":
        D = rec["code"].shape[-1]
        return codecs.q4_decode(rec["scale"], rec["code"].reshape(128, D // 32, 32))
    if fmt == "turbo3":
        D = rec["code"].shape[-1]
        return codecs.turbo3_decode(rec["scale"], rec["code"].reshape(128, D // 128, 128))
    if fmt == "tq5_0":
        D = rec["code"].shape[-1]
        return codecs.tq5_decode(rec["scale"], rec["code"].reshape(128, D // 128, 128))
    if fmt in QSYM:
        D = rec["code"].shape[-1]
        return codecs.qsym_decode(rec["scale"], rec["code"].reshape(128, D // 32, 32), QSYM[fmt])
    if fmt in QMIN:
        D = rec["code"].shape[-1]
        return codecs.qmin_decode(rec["scale"], rec["min"], rec["code"].reshape(128, D // 32, 32))
    if fmt.startswith("kvarn"):
        x = kvarn.decode(rec["code"], rec["S"], rec["Z"], rec["C"])   # [half, 128, 256]
        return x.transpose(1, 0, 2).reshape(128, -1)
    raise ValueError(fmt)


def pack_body(rec, fmt, role):
    """Unpacked record -> stored bytes (uint8 vector) for role 'K' or 'V'."""
    if fmt.startswith("kvarn"):
        parts = []
        for h in range(rec["code"].shape[0]):
            parts.append(kvarn.pack_codes(rec["code"][h], rec["bits"], role).reshape(-1))
            parts.append(kvarn.scale_block(rec["S"][h], rec["Z"][h], rec["C"][h]).view(np.uint8).reshape(-1))
        return np.concatenate(parts)
    code = rec["code"]                                   # [128 tokens, D]
    if fmt in ("turbo3", "tq5_0"):
        # token-major for K and V alike: turbo3 a 2-bit plane [128][D/4] then a one-bit plane
        # [128][D/8] of the 3-bit indices; tq5_0 the nibble plane [128][D/2] then a one-bit plane
        # [128][D/8]; then the fp16 norms (turbo3) or scales (tq5_0) [128][D/128]
        if fmt == "turbo3":
            parts = [codecs.pack_crumbs(code & 3).reshape(-1), codecs.pack_bitplane((code >> 2) & 1).reshape(-1)]
        else:
            parts = [codecs.pack_nibbles(code & 15).reshape(-1), codecs.pack_bitplane((code >> 4) & 1).reshape(-1)]
        parts.append(np.ascontiguousarray(rec["scale"]).astype(np.float16).view(np.uint8).reshape(-1))
        return np.concatenate(parts)
    if fmt in CODE_BITS:
        # token-major for K and V alike: the low nibble plane [128][D/2], the high plane (5-bit:
        # one bit per code [128][D/8]; 6-bit: two bits [128][D/4]), d [128][D/32], then for the
        # _1 formats m [128][D/32]
        parts = [codecs.pack_nibbles(code & 15).reshape(-1)]
        if CODE_BITS[fmt] == 5:
            parts.append(codecs.pack_bitplane((code >> 4) & 1).reshape(-1))
        elif CODE_BITS[fmt] == 6:
            parts.append(codecs.pack_crumbs((code >> 4) & 3).reshape(-1))
        parts.append(np.ascontiguousarray(rec["scale"]).astype(np.float16).view(np.uint8).reshape(-1))
        if fmt in QMIN:
            parts.append(np.ascontiguousarray(rec["min"]).astype(np.float16).view(np.uint8).reshape(-1))
        return np.concatenate(parts)
    rows = code if role == "K" else code.T               # K token-major, V channel-major
    if fmt in ("tbq4", "q4_0"):
        cb = codecs.pack_nibbles(rows)
    else:  # q8_0
        cb = rows.astype(np.int8).view(np.uint8)
    sc = np.ascontiguousarray(rec["scale"]).astype(np.float16).view(np.uint8)
    return np.concatenate([cb.reshape(-1), sc.reshape(-1)])


class HeadCache:
    """One (layer, sequence, KV head): sink, journal ring, exact tail, body records."""

    def __init__(self, cfg: HeadConfig):
        self.cfg = cfg
        D = cfg.head_dim
        self.N = 0
        self.S = SINK
        self.sink = {w: np.zeros((SINK, D), np.float16) for w in "KV"}
        if cfg.journal == "tq6_0":
            nb = D // 128
            self.jd = {w: np.zeros((cfg.ring, nb), np.float16) for w in "KV"}
            self.jcode = {w: np.zeros((cfg.ring, nb, 128), np.uint8) for w in "KV"}
            self.tail = {w: np.zeros((cfg.tail, D), np.uint16) for w in "KV"}
        else:
            self.jx = {w: np.zeros((cfg.ring, D), np.uint16) for w in "KV"}
        self.body = {w: [] for w in "KV"}

    # ------------------------------------------------------------------ append
    def append(self, k, v):
        """k, v: fp16 [n, D] for positions N .. N+n-1."""
        k = np.asarray(k, np.float16).reshape(-1, self.cfg.head_dim)
        v = np.asarray(v, np.float16).reshape(-1, self.cfg.head_dim)
        n = k.shape[0]
        if max(self.N + n, SINK) - self.S > self.cfg.ring:
            raise OverflowError("journal full")
        pos = np.arange(self.N, self.N + n)
        for w, x in (("K", k), ("V", v)):
            sink_m = pos < SINK
            self.sink[w][pos[sink_m]] = x[sink_m]
            jm = ~sink_m
            if not jm.any():
                continue
            pj, xj = pos[jm], x[jm]
            slot = (pj - SINK) % self.cfg.ring
            if self.cfg.journal == "tq6_0":
                y = rotate(xj.astype(np.float32), self.cfg.rot)
                d, code = codecs.tq6_encode(y)
                self.jd[w][slot] = d
                self.jcode[w][slot] = code
                self.tail[w][pj % self.cfg.tail] = _store_exact(xj, self.cfg.tail_fmt)
            else:
                self.jx[w][slot] = _store_exact(xj, self.cfg.journal)
        self.N += n

    # ------------------------------------------------------------------ seal
    def journal_rows(self, w, p0, n):
        """fp32 rows of positions [p0, p0+n) from the journal, in the body's domain."""
        slot = (np.arange(p0, p0 + n) - SINK) % self.cfg.ring
        if self.cfg.journal == "tq6_0":
            return codecs.tq6_decode(self.jd[w][slot], self.jcode[w][slot])
        x = _load_exact(self.jx[w][slot], self.cfg.journal)
        return rotate(x, self.cfg.rot)

    def seal(self, keep):
        """Seal every full group g with S + 128 <= N - keep; returns the count."""
        assert keep >= self.cfg.tail
        n = 0
        while self.S + GROUP <= self.N - keep:
            for w, fmt in (("K", self.cfg.k_body), ("V", self.cfg.v_body)):
                X = self.journal_rows(w, self.S, GROUP)
                self.body[w].append(encode_body(X, fmt, self.cfg.kvarn_balance))
            self.S += GROUP
            n += 1
        return n

    # ------------------------------------------------------------------ read
    def record_bytes(self, g, w):
        fmt = self.cfg.k_body if w == "K" else self.cfg.v_body
        return pack_body(self.body[w][g], fmt, w)

    def tq6_slot_bytes(self, p, w):
        """(d fp16 [nb], ql [nb, 64], qh [nb, 32]) of the journal slot of position p."""
        slot = (p - SINK) % self.cfg.ring
        ql, qh = codecs.tq6_pack(self.jcode[w][slot])
        return self.jd[w][slot], ql, qh

    def regions(self):
        """[(domain, K [n, D] fp32, V [n, D] fp32)] covering positions [0, N) once."""
        N, S, cfg = self.N, self.S, self.cfg
        out = []
        ns = min(N, SINK)
        out.append(("exact", self.sink["K"][:ns].astype(np.float32), self.sink["V"][:ns].astype(np.float32)))
        if S > SINK:
            Kb = np.concatenate([decode_body(r, cfg.k_body) for r in self.body["K"]])
            Vb = np.concatenate([decode_body(r, cfg.v_body) for r in self.body["V"]])
            out.append(("rot", Kb, Vb))
        if N > S:
            if cfg.journal == "tq6_0":
                E = max(S, N - cfg.tail)
                if E > S:
                    out.append(("rot", self.journal_rows("K", S, E - S), self.journal_rows("V", S, E - S)))
                pos = np.arange(E, N) % cfg.tail
                out.append(("exact", _load_exact(self.tail["K"][pos], cfg.tail_fmt),
                            _load_exact(self.tail["V"][pos], cfg.tail_fmt)))
            else:
                slot = (np.arange(S, N) - SINK) % cfg.ring
                out.append(("exact", _load_exact(self.jx["K"][slot], cfg.journal),
                            _load_exact(self.jx["V"][slot], cfg.journal)))
        return out
