"""Seeded synthetic inputs for the CSA2 layer.

This module is the one place both the CUDA path and the CPU oracle take their
inputs from.  It holds none of the layer's arithmetic (no scoring, selection,
visibility rule, softmax or tail rule): it draws N(0,1) tensors from seeded
torch generators, encodes them into the storage formats the layer reads, and
lays out the workloads' structure (requests, positions, pool rows) exactly as
each workload states it.

Storage formats produced (the producer side of the layer, used here only to
synthesise inputs):
  * index operands: MXFP4 -- E2M1 codes, two per byte (element 2i in the low
    nibble), one power-of-two fp32 scale per 32 elements, chosen as in the OCP
    MX recipe (scale = 2^(floor(log2 amax) - 2), elements clamped to +-6);
  * KV and SWA rows: E4M3 codes with one fp32 scale per 32 channels
    (scale = amax / 448, 1 for an all-zero block);
  * queries: bf16.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Dict, List, Optional, Tuple

import torch

DIM = 512          # shared latent KV row width
IDX_DIM = 128      # index head width
TOPK = 512
WINDOW = 128
BLOCK = 8
MAX_BLOCKS = 2048

# E2M1 magnitudes in code order 0..7 and the midpoints used to round onto them
_E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
_E2M1_MID = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)

_CHUNK_ROWS = 1 << 18


def generator(seed: int, tensor_id: str, device) -> torch.Generator:
    """A torch generator keyed by (seed, tensor_id)."""
    h = hashlib.sha256(f"{seed}:{tensor_id}".encode()).digest()
    g = torch.Generator(device=device)
    g.manual_seed(int.from_bytes(h[:8], "little") & ((1 << 63) - 1))
    return g


def randn(shape, seed: int, tensor_id: str, device="cpu") -> torch.Tensor:
    return torch.randn(shape, generator=generator(seed, tensor_id, device),
                       device=device, dtype=torch.float32)


def uniform(shape, seed: int, tensor_id: str, device="cpu") -> torch.Tensor:
    return torch.rand(shape, generator=generator(seed, tensor_id, device),
                      device=device, dtype=torch.float64)


# --------------------------------------------------------------------------
# encoders (input synthesis only)
# --------------------------------------------------------------------------

def encode_mxfp4(x: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """x [..., D] float32 -> (codes uint8 [..., D/2], scales float32 [..., D/32])."""
    d = x.shape[-1]
    g = x.reshape(*x.shape[:-1], d // 32, 32)
    amax = g.abs().amax(-1, keepdim=True)
    expo = torch.floor(torch.log2(amax.clamp_min(2.0 ** -100))) - 2
    scale = torch.where(amax > 0, torch.exp2(expo), torch.ones_like(amax))
    y = (g / scale).clamp(-6.0, 6.0)
    mid = torch.tensor(_E2M1_MID, device=x.device, dtype=torch.float32)
    mag_code = torch.bucketize(y.abs(), mid).to(torch.uint8)
    code = mag_code | ((y < 0) & (mag_code > 0)).to(torch.uint8) << 3
    code = code.reshape(*x.shape[:-1], d)
    packed = code[..., 0::2] | (code[..., 1::2] << 4)
    return packed.contiguous(), scale.reshape(*x.shape[:-1], d // 32).contiguous()


def encode_fp8_block32(x: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """x [..., D] float32 -> (E4M3 codes uint8 [..., D], scales float32 [..., D/32])."""
    d = x.shape[-1]
    g = x.reshape(*x.shape[:-1], d // 32, 32)
    amax = g.abs().amax(-1, keepdim=True)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    y = (g / scale).clamp(-448.0, 448.0)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(*x.shape[:-1], d)
    return codes.contiguous(), scale.reshape(*x.shape[:-1], d // 32).contiguous()


def encode_fp4kv(x: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """x [..., D] float32 -> (E2M1 codes uint8 [..., D/2], E4M3 scale codes
    uint8 [..., D/16]): the main-KV FP4 layout, one E4M3 scale per 16 channels
    (amax/6 rounded to E4M3, no second-level global scale), elements x/scale
    clamped to +-6 and rounded to the E2M1 grid; element 2i in the low nibble."""
    d = x.shape[-1]
    g = x.reshape(*x.shape[:-1], d // 16, 16)
    amax = g.abs().amax(-1, keepdim=True)
    sc = (amax / 6.0).clamp(max=448.0).to(torch.float8_e4m3fn)
    s = sc.to(torch.float32)
    y = torch.where(s > 0, g / torch.where(s > 0, s, torch.ones_like(s)), torch.zeros_like(g))
    y = y.clamp(-6.0, 6.0)
    mid = torch.tensor(_E2M1_MID, device=x.device, dtype=torch.float32)
    mag_code = torch.bucketize(y.abs(), mid).to(torch.uint8)
    code = mag_code | ((y < 0) & (mag_code > 0)).to(torch.uint8) << 3
    code = code.reshape(*x.shape[:-1], d)
    packed = code[..., 0::2] | (code[..., 1::2] << 4)
    return packed.contiguous(), sc.view(torch.uint8).reshape(*x.shape[:-1], d // 16).contiguous()


def fp8_rows(n: int, seed: int, tensor_id: str, device, dim: int = DIM):
    """n N(0,1) rows encoded as E4M3 block-32 (generated in chunks)."""
    codes = torch.empty((n, dim), dtype=torch.uint8, device=device)
    scales = torch.empty((n, dim // 32), dtype=torch.float32, device=device)
    for c0 in range(0, n, _CHUNK_ROWS):
        c1 = min(n, c0 + _CHUNK_ROWS)
        x = randn((c1 - c0, dim), seed, f"{tensor_id}/{c0}", device)
        codes[c0:c1], scales[c0:c1] = encode_fp8_block32(x)
    return codes, scales


def fp4kv_rows(n: int, seed: int, tensor_id: str, device, dim: int = DIM):
    """The same N(0,1) rows as fp8_rows(n, seed, tensor_id) in the FP4 main-KV layout."""
    codes = torch.empty((n, dim // 2), dtype=torch.uint8, device=device)
    sf = torch.empty((n, dim // 16), dtype=torch.uint8, device=device)
    for c0 in range(0, n, _CHUNK_ROWS):
        c1 = min(n, c0 + _CHUNK_ROWS)
        x = randn((c1 - c0, dim), seed, f"{tensor_id}/{c0}", device)
        codes[c0:c1], sf[c0:c1] = encode_fp4kv(x)
    return codes, sf


def fp4_rows(n: int, seed: int, tensor_id: str, device, dim: int = IDX_DIM):
    """n N(0,1) rows encoded as MXFP4 (generated in chunks)."""
    codes = torch.empty((n, dim // 2), dtype=torch.uint8, device=device)
    scales = torch.empty((n, dim // 32), dtype=torch.float32, device=device)
    for c0 in range(0, n, _CHUNK_ROWS):
        c1 = min(n, c0 + _CHUNK_ROWS)
        x = randn((c1 - c0, dim), seed, f"{tensor_id}/{c0}", device)
        codes[c0:c1], scales[c0:c1] = encode_mxfp4(x)
    return codes, scales


# --------------------------------------------------------------------------
# workload structure
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Pool:
    """The KV-source layer's shared pool: compressed KV rows and index keys."""
    kv_fp8: torch.Tensor      # [Nkv, 512] uint8
    kv_scale: torch.Tensor    # [Nkv, 16] f32
    k_fp4: torch.Tensor       # [Nkv, 64] uint8
    k_scale: torch.Tensor     # [Nkv, 4] f32
    kv_start: torch.Tensor    # [R] int64
    kv_len: torch.Tensor      # [R] int64
    tag: str = ""             # generator stream of the rows
    kv_fp4: Optional[torch.Tensor] = None   # [Nkv, 256] uint8 E2M1 (FP4 main-KV layout)
    kv_sf: Optional[torch.Tensor] = None    # [Nkv, 32] uint8 E4M3 scale per 16 channels


@dataclasses.dataclass
class Layer:
    """One consumer layer's own tensors: queries, index queries, SWA rows."""
    name: str
    mode: str                          # "full" | "source" | "reindex" | "reuse"
    q: torch.Tensor                    # [Nq, H, 512] bf16
    swa_fp8: torch.Tensor              # [Nswa, 512] uint8
    swa_scale: torch.Tensor            # [Nswa, 16] f32
    swa_start: torch.Tensor            # [R] int64
    swa_pos0: torch.Tensor             # [R] int64
    swa_len: torch.Tensor              # [R] int64
    win_lo: Optional[torch.Tensor]     # [Nq] int64 or None (normal window)
    q_fp4: Optional[torch.Tensor] = None     # [Nq, Hi, 64] uint8
    q_scale: Optional[torch.Tensor] = None   # [Nq, Hi, 4] f32
    head_w: Optional[torch.Tensor] = None    # [Nq, Hi] f32
    given_idx: Optional[torch.Tensor] = None  # [Nq, K] int32 (Reuse with external indices)


@dataclasses.dataclass
class Workload:
    name: str
    ratio: int
    n_heads: int
    n_idx_heads: int
    q_req: torch.Tensor        # [Nq] int32
    q_pos: torch.Tensor        # [Nq] int64
    pool: Pool
    layers: Dict[str, Layer]
    topk: int = TOPK
    window: int = WINDOW
    replay: int = WINDOW       # rows kept per request by the tail layout (R)
    block: int = BLOCK
    max_blocks: int = MAX_BLOCKS
    extend_len: Optional[torch.Tensor] = None   # [R] int32 when the rows are tails
    seq_len: Optional[torch.Tensor] = None      # [R] int64
    ld: int = 0                                 # score row capacity (full mode)
    notes: str = ""

    @property
    def num_q(self) -> int:
        return int(self.q_pos.shape[0])

    @property
    def num_req(self) -> int:
        return int(self.pool.kv_start.shape[0])

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(DIM)

    def batch(self, layer: str, rows: Optional[torch.Tensor] = None) -> dict:
        """The batch description of ``layer`` (optionally restricted to query
        rows ``rows``) as a dict of tensors on the workload's device."""
        L = self.layers[layer]
        q_req, q_pos = self.q_req, self.q_pos
        if rows is not None:
            q_req, q_pos = q_req[rows], q_pos[rows]
        return dict(num_q=int(q_pos.shape[0]), num_req=self.num_req, ratio=self.ratio,
                    q_req=q_req, q_pos=q_pos, kv_start=self.pool.kv_start,
                    kv_len=self.pool.kv_len, swa_start=L.swa_start,
                    swa_pos0=L.swa_pos0, swa_len=L.swa_len)


def _i64(v, device):
    return torch.as_tensor(v, dtype=torch.int64).to(device)


def _i32(v, device):
    return torch.as_tensor(v, dtype=torch.int32).to(device)


def make_pool(entries: List[int], seed: int, tag: str, device) -> Pool:
    starts, s = [], 0
    for n in entries:
        starts.append(s)
        s += int(n)
    kv_fp8, kv_scale = fp8_rows(s, seed, f"{tag}/kv", device)
    k_fp4, k_scale = fp4_rows(s, seed, f"{tag}/k", device)
    return Pool(kv_fp8, kv_scale, k_fp4, k_scale, _i64(starts, device), _i64(entries, device),
                tag)


def with_fp4kv(w: "Workload", seed: int = 0) -> "Workload":
    """Add the FP4 main-KV encoding of the workload's pool rows (the same
    underlying N(0,1) rows as its FP8 pool)."""
    p = w.pool
    p.kv_fp4, p.kv_sf = fp4kv_rows(p.kv_fp8.shape[0], seed, f"{p.tag}/kv", p.kv_fp8.device)
    return w


def make_layer(name: str, mode: str, nq: int, n_heads: int, n_idx_heads: int,
               swa_ranges: List[Tuple[int, int]], win_lo, seed: int, tag: str, device,
               with_index: bool) -> Layer:
    """``swa_ranges`` = per request (first absolute position held, rows held)."""
    q = randn((nq, n_heads, DIM), seed, f"{tag}/{name}/q", device).to(torch.bfloat16)
    total = sum(n for _, n in swa_ranges)
    swa_fp8, swa_scale = fp8_rows(max(total, 1), seed, f"{tag}/{name}/swa", device)
    starts, s = [], 0
    for _, n in swa_ranges:
        starts.append(s)
        s += n
    L = Layer(name, mode, q, swa_fp8, swa_scale, _i64(starts, device),
              _i64([p for p, _ in swa_ranges], device), _i64([n for _, n in swa_ranges], device),
              None if win_lo is None else _i64(win_lo, device))
    if with_index:
        x = randn((nq, n_idx_heads, IDX_DIM), seed, f"{tag}/{name}/qi", device)
        L.q_fp4, L.q_scale = encode_mxfp4(x)
        L.head_w = randn((nq, n_idx_heads), seed, f"{tag}/{name}/w", device) / math.sqrt(n_idx_heads)
    return L


# --------------------------------------------------------------------------
# generic shapes (the five workloads below and the scaled-down test cases)
# --------------------------------------------------------------------------

def full_layer(ctx: int, ratio: int, q_positions: List[int], n_heads: int, n_idx_heads: int,
               seed: int = 0, device="cpu", tail_win_lo: Optional[int] = None,
               tag: str = "full", topk: int = TOPK) -> Workload:
    """One request of ``ctx`` tokens, compressed ``ratio``:1 into ctx // ratio
    entries, queried at ``q_positions``; a Full layer (own scoring and top-K)
    whose SWA holds every position the queries' windows reach."""
    entries = ctx // ratio
    pool = make_pool([entries], seed, tag, device)
    lo = max(0, min(q_positions) - WINDOW + 1)
    hi = max(q_positions) + 1
    nq = len(q_positions)
    win_lo = None if tail_win_lo is None else [tail_win_lo] * nq
    L = make_layer("full", "full", nq, n_heads, n_idx_heads, [(lo, hi - lo)], win_lo,
                   seed, tag, device, True)
    return Workload(tag, ratio, n_heads, n_idx_heads, _i32([0] * nq, device),
                    _i64(q_positions, device), pool, {"full": L}, topk=topk, ld=entries)


def decoder_replay(extends: List[int], prefixes: List[int], n_heads: int, n_idx_heads: int,
                   seed: int = 0, device="cpu", tag: str = "replay",
                   topk: int = TOPK, max_blocks: int = MAX_BLOCKS, block: int = BLOCK,
                   replay: int = WINDOW) -> Workload:
    """Requests r = 0.. each with an extend of ``extends[r]`` tokens over
    ``prefixes[r]`` cached tokens (m = 1: one compressed entry per token).  The
    query rows are each request's bounded-replay tail: the last
    min(replay, extend) rows at their absolute positions (replay = R, 128 in
    the fixed build; other budgets are the R sweep of "SGLang 如何让 DeepSeek
    V4.1 Flash 的后半层只处理尾部 token" sec. 3.5, with the SWA width kept at 128).  Layers: an L20-style
    source pass over those rows (normal window, full-visible scoring, top-K and
    candidate pool), an L21-style Reindex layer (pool-restricted scoring, tail
    window) and an L22-style Reuse layer (tail window, the Reindex layer's
    indices)."""
    n_req = len(extends)
    seqs = [p + e for p, e in zip(prefixes, extends)]
    tails = [min(replay, e) for e in extends]
    q_req, q_pos, win = [], [], []
    for r in range(n_req):
        q_req += [r] * tails[r]
        q_pos += list(range(seqs[r] - tails[r], seqs[r]))
        win += [seqs[r] - tails[r]] * tails[r]
    pool = make_pool(seqs, seed, tag, device)
    nq = len(q_pos)
    src = [(max(0, s - t - WINDOW + 1), s - max(0, s - t - WINDOW + 1)) for s, t in zip(seqs, tails)]
    late = [(s - t, t) for s, t in zip(seqs, tails)]
    L20 = make_layer("L20", "source", nq, n_heads, n_idx_heads, src, None, seed, tag, device, True)
    L21 = make_layer("L21", "reindex", nq, n_heads, n_idx_heads, late, win, seed, tag, device, True)
    L22 = make_layer("L22", "reuse", nq, n_heads, n_idx_heads, late, win, seed, tag, device, False)
    return Workload(tag, 1, n_heads, n_idx_heads, _i32(q_req, device), _i64(q_pos, device), pool,
                    {"L20": L20, "L21": L21, "L22": L22}, topk=topk, block=block,
                    max_blocks=max_blocks, replay=replay, extend_len=_i32(extends, device),
                    seq_len=_i64(seqs, device), ld=max(seqs))


def hierarchical(ctx: int, nq: int, n_heads: int, n_idx_heads: int, seed: int = 0,
                 device="cpu", tag: str = "hier", max_blocks: int = MAX_BLOCKS,
                 block: int = BLOCK, topk: int = TOPK) -> Workload:
    """One request of ``ctx`` tokens at m = 1, queried at its last ``nq``
    positions with normal windows: an L20-style source (full scoring, own
    top-K, candidate pool) and the next index source restricted to that pool."""
    pool = make_pool([ctx], seed, tag, device)
    q_pos = list(range(ctx - nq, ctx))
    lo = max(0, ctx - nq - WINDOW + 1)
    src = make_layer("L20", "source", nq, n_heads, n_idx_heads, [(lo, ctx - lo)], None,
                     seed, tag, device, True)
    con = make_layer("L21", "reindex", nq, n_heads, n_idx_heads, [(lo, ctx - lo)], None,
                     seed, tag, device, True)
    return Workload(tag, 1, n_heads, n_idx_heads, _i32([0] * nq, device), _i64(q_pos, device),
                    pool, {"L20": src, "L21": con}, topk=topk, block=block,
                    max_blocks=max_blocks, ld=ctx)


def ragged_mixed(n_decode: int, n_extend: int, extend: int, ctx_lo: int, ctx_hi: int,
                 n_heads: int, n_idx_heads: int, seed: int = 0, device="cpu",
                 tag: str = "ragged", topk: int = TOPK) -> Workload:
    """``n_decode`` decode requests (one query at t = C - 1, C log-uniform in
    [ctx_lo, ctx_hi)) and ``n_extend`` short extends of ``extend`` tokens over
    prefixes drawn from the same law (window truncated to the extend: tail
    rows with lower bound S - E).  m = 1.  Even request ids run a Reindex
    layer over all visible entries, odd ids a Reuse layer whose indices are a
    uniform sample without replacement of min(K, t+1) entries at positions <= t."""
    u = uniform((n_decode + n_extend,), seed, f"{tag}/ctx")
    ctx = [int(math.floor(ctx_lo * (ctx_hi / ctx_lo) ** float(v))) for v in u]
    entries, q_req, q_pos, win_lo, swa = [], [], [], [], []
    for r in range(n_decode):
        c = ctx[r]
        entries.append(c)
        q_req.append(r)
        q_pos.append(c - 1)
        win_lo.append(0)
        swa.append((max(0, c - WINDOW), min(c, WINDOW)))
    ext_len, seq_len = [], []
    for e in range(n_extend):
        r = n_decode + e
        p = ctx[r]
        s = p + extend
        entries.append(s)
        ext_len.append(extend)
        seq_len.append(s)
        for k in range(extend):
            q_req.append(r)
            q_pos.append(p + k)
            win_lo.append(p)
        swa.append((p, extend))
    pool = make_pool(entries, seed, tag, device)
    nq = len(q_pos)
    L = make_layer("mixed", "mixed", nq, n_heads, n_idx_heads, swa, win_lo, seed, tag, device, True)
    # Reuse rows: indices handed over from an earlier index source
    g = generator(seed, f"{tag}/reuse", "cpu")
    given = torch.full((nq, topk), -1, dtype=torch.int32)
    for i in range(nq):
        if q_req[i] % 2 == 1:
            n = q_pos[i] + 1
            take = min(topk, n)
            if n <= 4 * topk:
                pick = torch.randperm(n, generator=g)[:take]
            else:
                pick = torch.unique(torch.randint(0, n, (3 * take,), generator=g))
                pick = pick[torch.randperm(pick.numel(), generator=g)][:take]
            given[i, :take] = pick.to(torch.int32)
    L.given_idx = given.to(device)
    return Workload(tag, 1, n_heads, n_idx_heads, _i32(q_req, device), _i64(q_pos, device), pool,
                    {"mixed": L}, topk=topk, ld=max(entries),
                    extend_len=_i32([0] * n_decode + ext_len, device),
                    seq_len=_i64([c for c in ctx[:n_decode]] + seq_len, device))


# --------------------------------------------------------------------------
# the five named workloads
# --------------------------------------------------------------------------

CONFIG_NAMES = ("c1_tiny_full", "c2_decoder_replay", "c3_encoder_prefill",
                "c4_hierarchical", "c5_ragged_mixed")


def config(name: str, device="cpu", seed: int = 0) -> Workload:
    if name == "c1_tiny_full":
        w = full_layer(4096, 2, list(range(3968, 4096)), 16, 8, seed, device, tag=name)
    elif name == "c2_decoder_replay":
        w = decoder_replay([8192] * 8, [0] * 8, 64, 32, seed, device, tag=name)
    elif name == "c3_encoder_prefill":
        w = full_layer(32768, 2, list(range(32768)), 64, 32, seed, device, tag=name)
    elif name == "c4_hierarchical":
        w = hierarchical(131072, 512, 64, 32, seed, device, tag=name)
    elif name == "c5_ragged_mixed":
        w = ragged_mixed(256, 16, 64, 4096, 524288, 64, 32, seed, device, tag=name)
    else:
        raise KeyError(name)
    w.name = name
    return w
