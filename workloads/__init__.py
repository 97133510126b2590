"""Seeded synthetic workloads for sparse MLA decode.

This module only draws random numbers and lays them out in the shapes the
decode consumes. It holds none of the method's arithmetic: no quantisation,
no index translation, no attention. The float64 oracle and the CUDA path both
take their inputs from here; neither imports the other.

Shapes follow the DeepSeek-V3.2/V4 sparse-MLA decode setting the source pages
describe (vLLM PR #43477 "实现拆解" and "关键源码片段": one shared 576-dim latent
per slot, a paged cache, request-local top-k indices padded with -1, output
[tokens, heads, 512]). What is drawn, and how:

* context lengths: uniform integers in [ctx_lo, ctx_hi] per request;
* physical pages: one shuffled permutation of the whole pool, cut into each
  request's page list (so neighbouring logical pages are far apart in HBM);
* top-k indices: for query token i of a request with next_n query tokens, the
  visible context is ctx - (next_n - 1) + i; min(visible, topk - tail_pad)
  distinct indices are drawn uniformly from it, in random order, and the
  rest of the row is -1;
* q ~ N(0, 1) rounded to bf16; sink ~ N(0, 1) fp32 per head;
* cache source values ~ N(0, 1) rounded to bf16: 512 latent + 64 RoPE per
  slot. For the bf16 cache format these ARE the cache rows. For the FP8
  format they are the values each side quantises itself (the CUDA path with
  its pack kernel, the oracle with its own packer).
* optional magnitude sweeps for operand-range tests: a gain per head on q
  (q_gains, cycled over heads), per dimension on q (q_dim_gains, cycled over
  the 576 dims), and per physical slot on the latent and RoPE source values
  (latent_gains / rope_gains, cycled over slots); each multiplies the N(0, 1)
  draw in fp32 before the rounding to bf16.

Large pools are produced in chunks of CHUNK_SLOTS slots, each from its own
seeded generator, so any chunk can be regenerated on its own.
"""
from __future__ import annotations

import dataclasses
import math

import torch

SEED_BASE = 20261202
CHUNK_SLOTS = 1 << 20
LATENT_DIM = 512
ROPE_DIM = 64
HEAD_DIM = LATENT_DIM + ROPE_DIM
# fp32 value of 1/sqrt(576) (= 1/24 rounded to fp32)
SM_SCALE_576 = float(torch.tensor(1.0 / math.sqrt(HEAD_DIM), dtype=torch.float32).item())


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_requests: int
    next_n: int
    num_heads: int
    topk: int
    page_size: int
    kv_format: str  # "bf16" (1152 B per slot), "fp8_ds" (656 B) or "fp8_tensor" (576 B)
    ctx_lo: int
    ctx_hi: int
    sink: bool
    tail_pad: int = 0  # trailing -1 entries forced into every index row
    shared_pool_pages: int = 0  # > 0: every request maps the same small pool
    sm_scale: float = SM_SCALE_576
    seed_offset: int = 0
    kv_scale: float = 1.0  # per-tensor scale of the fp8_tensor format (unused otherwise)
    q_gains: tuple = ()       # per-head multipliers of q (cycled), empty = 1
    q_dim_gains: tuple = ()   # per-dim multipliers of q (cycled over 576 dims), empty = 1
    latent_gains: tuple = ()  # per-slot multipliers of the latent source values (cycled)
    rope_gains: tuple = ()    # per-slot multipliers of the RoPE source values (cycled)

    @property
    def num_tokens(self) -> int:
        return self.num_requests * self.next_n

    @property
    def row_bytes(self) -> int:
        return {"fp8_ds": 656, "fp8_tensor": HEAD_DIM}.get(self.kv_format, 2 * HEAD_DIM)

    @property
    def page_table_stride(self) -> int:
        if self.shared_pool_pages:
            return self.shared_pool_pages
        return -(-self.ctx_hi // self.page_size)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five decode workloads, smallest first.
WORKLOADS = [
    # 2 requests x 1 token, 16 heads, top-k 128 of a 256-slot bf16 pool
    # (4 pages x 64 slots, both requests map all 4 pages in shuffled order).
    Workload("tiny_bf16_T2_H16_K128", 2, 1, 16, 128, 64, "bf16", 256, 256, False,
             shared_pool_pages=4, seed_offset=0),
    # 32 requests x 1 token, 64 heads, context U[1k, 32k], -1 padded below 2048.
    Workload("fp8_T32_H64_K2048_ctx1k-32k", 32, 1, 64, 2048, 64, "fp8_ds", 1024, 32768,
             False, seed_offset=1),
    # 128 requests x 1 token, 128 heads, 64k context each, per-head sink.
    Workload("fp8_T128_H128_K2048_ctx64k_sink", 128, 1, 128, 2048, 64, "fp8_ds", 65536, 65536,
             True, seed_offset=2),
    # MTP: 64 requests x 4 query tokens with independent index sets, 128 heads, sink.
    Workload("fp8_mtp_T256_H128_K2048_ctx4k-128k_sink", 64, 4, 128, 2048, 64, "fp8_ds", 4096,
             131072, True, seed_offset=3),
    # 256 requests x 1 token, 16 heads (one tensor-parallel head shard), last 410 of
    # 2048 indices are -1 (20% tail padding).
    Workload("fp8_T256_H16_K2048_ctx8k-128k_pad20", 256, 1, 16, 2048, 64, "fp8_ds", 8192,
             131072, False, tail_pad=410, seed_offset=4),
]
# The per-tensor FP8 cache of the FlashInfer path (vLLM PR #43827): the default
# workload's batch with that format, at the per-tensor scale 1.0 the page's code uses.
EXTRA_WORKLOADS = [
    Workload("fp8tensor_T32_H64_K2048_ctx1k-32k", 32, 1, 64, 2048, 64, "fp8_tensor", 1024, 32768,
             False, seed_offset=5, kv_scale=1.0),
    # the two 128-head batches on the per-tensor cache, for FP8 q against it
    Workload("fp8tensor_T128_H128_K2048_ctx64k_sink", 128, 1, 128, 2048, 64, "fp8_tensor", 65536, 65536,
             True, seed_offset=6, kv_scale=1.0),
    Workload("fp8tensor_mtp_T256_H128_K2048_ctx4k-128k_sink", 64, 4, 128, 2048, 64, "fp8_tensor", 4096,
             131072, True, seed_offset=7, kv_scale=1.0),
]
# Per-tensor scale of FP8 q in the tests and the bench: N(0, 1) q maps to |q / 2^-5| < 448.
Q_SCALE_FP8 = 2.0 ** -5


def q_to_e4m3(q: torch.Tensor, q_scale: float = Q_SCALE_FP8) -> torch.Tensor:
    """The caller's FP8 q: E4M3FN codes (uint8, same shape) of q / q_scale by torch's cast,
    clamped to +-448 first (an input of the decode, like q itself)."""
    x = (q.float() / q_scale).clamp(-448.0, 448.0)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)
BY_NAME = {w.name: w for w in WORKLOADS + EXTRA_WORKLOADS}


def _mix(seed: int, tag: int) -> int:
    return (seed * 0x9E3779B1 + tag * 0x85EBCA77 + 0x165667B1) % (1 << 62)


def _gen(seed: int, tag: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_mix(seed, tag))
    return g


@dataclasses.dataclass
class Problem:
    """One drawn decode batch. Tensors live on `device`."""

    w: Workload
    seed: int
    device: torch.device
    ctx: torch.Tensor  # [B] int64 context length per request
    page_table: torch.Tensor  # [B, stride] int32, unused entries -1
    num_pages: int
    topk: torch.Tensor  # [T, K] int32 request-local slot ids, -1 = padding
    q: torch.Tensor  # [T, H, 576] bf16
    sink: torch.Tensor | None  # [H] fp32
    kv_bf16: torch.Tensor | None  # [num_pages, P, 576] bf16 (bf16 format only)

    @property
    def num_slots(self) -> int:
        return self.num_pages * self.w.page_size

    @property
    def num_chunks(self) -> int:
        return -(-self.num_slots // CHUNK_SLOTS)

    def raw_chunk(self, c: int, device=None):
        """Source values of physical slots [c*CHUNK_SLOTS, ...): (latent [n,512], rope [n,64]) bf16."""
        dev = self.device if device is None else device
        lo = c * CHUNK_SLOTS
        n = min(CHUNK_SLOTS, self.num_slots - lo)
        g = _gen(self.seed, 1000 + c, dev)
        x = torch.randn((n, HEAD_DIM), generator=g, device=dev, dtype=torch.float32)
        for gains, cols in ((self.w.latent_gains, slice(0, LATENT_DIM)), (self.w.rope_gains, slice(LATENT_DIM, None))):
            if gains:
                gt = torch.tensor(gains, dtype=torch.float32, device=dev)
                slot = torch.arange(lo, lo + n, device=dev) % len(gains)
                x[:, cols] *= gt[slot][:, None]
        x = x.to(torch.bfloat16)
        return x[:, :LATENT_DIM].contiguous(), x[:, LATENT_DIM:].contiguous()

    def raw_pages(self, pages) -> tuple[torch.Tensor, torch.Tensor]:
        """Source values of whole physical pages (sorted, unique), on the host.

        Returns (latent [len(pages)*P, 512], rope [len(pages)*P, 64]) bf16, rows in
        the order of `pages`, each page's P slots in order.
        """
        P = self.w.page_size
        pages = sorted(set(int(p) for p in pages))
        lat_out = torch.empty((len(pages) * P, LATENT_DIM), dtype=torch.bfloat16)
        rope_out = torch.empty((len(pages) * P, ROPE_DIM), dtype=torch.bfloat16)
        by_chunk: dict[int, list[tuple[int, int]]] = {}
        for i, p in enumerate(pages):
            by_chunk.setdefault((p * P) // CHUNK_SLOTS, []).append((i, p))
        for c, items in by_chunk.items():
            lat, rope = self.raw_chunk(c)
            for i, p in items:
                s = p * P - c * CHUNK_SLOTS
                lat_out[i * P:(i + 1) * P] = lat[s:s + P].cpu()
                rope_out[i * P:(i + 1) * P] = rope[s:s + P].cpu()
        return lat_out, rope_out


def make_problem(w: Workload, seed: int | None = None, device="cpu") -> Problem:
    device = torch.device(device)
    if seed is None:
        seed = SEED_BASE + w.seed_offset
    B, T, H, K, P = w.num_requests, w.num_tokens, w.num_heads, w.topk, w.page_size
    stride = w.page_table_stride

    # context lengths
    if w.shared_pool_pages:
        ctx = torch.full((B,), w.shared_pool_pages * P, dtype=torch.int64)
    elif w.ctx_lo == w.ctx_hi:
        ctx = torch.full((B,), w.ctx_lo, dtype=torch.int64)
    else:
        ctx = torch.randint(w.ctx_lo, w.ctx_hi + 1, (B,), generator=_gen(seed, 1, "cpu"))

    # page table: shuffled physical pages
    page_table = torch.full((B, stride), -1, dtype=torch.int32)
    if w.shared_pool_pages:
        num_pages = w.shared_pool_pages
        for r in range(B):
            page_table[r] = torch.randperm(num_pages, generator=_gen(seed, 200 + r, "cpu")).to(torch.int32)
    else:
        npages = [-(-int(c) // P) for c in ctx]
        num_pages = sum(npages)
        perm = torch.randperm(num_pages, generator=_gen(seed, 2, "cpu")).to(torch.int32)
        off = 0
        for r in range(B):
            page_table[r, :npages[r]] = perm[off:off + npages[r]]
            off += npages[r]

    # top-k indices: distinct, random order, -1 tail
    topk = torch.full((T, K), -1, dtype=torch.int32)
    g = _gen(seed, 3, device)
    for t in range(T):
        r, i = divmod(t, w.next_n)
        visible = int(ctx[r]) - (w.next_n - 1) + i
        nvalid = min(visible, K - w.tail_pad)
        idx = torch.randperm(visible, generator=g, device=device)[:nvalid]
        topk[t, :nvalid] = idx.to(torch.int32).cpu()

    q = torch.randn((T, H, HEAD_DIM), generator=_gen(seed, 4, device), device=device,
                    dtype=torch.float32)
    if w.q_gains:
        qg = torch.tensor(w.q_gains, dtype=torch.float32, device=device)
        q *= qg[torch.arange(H, device=device) % len(w.q_gains)][None, :, None]
    if w.q_dim_gains:
        dg = torch.tensor(w.q_dim_gains, dtype=torch.float32, device=device)
        q *= dg[torch.arange(HEAD_DIM, device=device) % len(w.q_dim_gains)][None, None, :]
    q = q.to(torch.bfloat16)
    sink = None
    if w.sink:
        sink = torch.randn((H,), generator=_gen(seed, 5, device), device=device, dtype=torch.float32)
    kv_bf16 = None
    if w.kv_format == "bf16":
        x = torch.randn((num_pages * P, HEAD_DIM), generator=_gen(seed, 6, device), device=device,
                        dtype=torch.float32)
        kv_bf16 = x.to(torch.bfloat16).view(num_pages, P, HEAD_DIM)

    return Problem(w=w, seed=seed, device=device, ctx=ctx, page_table=page_table.to(device),
                   num_pages=num_pages, topk=topk.to(device), q=q, sink=sink, kv_bf16=kv_bf16)


def small_variant(w: Workload, num_requests: int, ctx_lo: int, ctx_hi: int, topk: int,
                  tail_pad: int = 0, name_suffix: str = "small") -> Workload:
    """A reduced copy of a workload (same heads, format, sink, next_n) for oracle-speed tests."""
    return w.replace(name=f"{w.name}:{name_suffix}", num_requests=num_requests, ctx_lo=ctx_lo,
                     ctx_hi=ctx_hi, topk=topk, tail_pad=tail_pad, shared_pool_pages=0)


# ------------------------------------------------------------------------------ indexer inputs

INDEX_HEADS = 64
INDEX_DIM = 128


@dataclasses.dataclass
class IndexerInputs:
    """Inputs of the sparse-attention indexer for a decode batch (same requests and pages).

    q [T, H_I, 128] E4M3 codes (uint8); weights [T, H_I] fp32; cache [num_pages, P * 132]
    bytes, each page P x 128 E4M3 key codes (slot-major) followed by P fp32 key scales;
    ctx [B] int32 context lengths. The codes are drawn as N(0, 1) values (q) and
    N(0, 1) * 32 values (keys) cast to float8_e4m3fn by torch; the key scales are powers of
    two 2^e with e uniform in [-10, -4]; the weights are N(0, 1) / 8.
    """

    q: torch.Tensor
    weights: torch.Tensor
    cache: torch.Tensor
    ctx: torch.Tensor
    heads: int = INDEX_HEADS


def make_indexer_inputs(problem: Problem, seed: int | None = None, heads: int = INDEX_HEADS,
                        device=None) -> IndexerInputs:
    dev = problem.device if device is None else torch.device(device)
    seed = problem.seed if seed is None else seed
    w = problem.w
    T, P = w.num_tokens, w.page_size
    q = torch.randn((T, heads, INDEX_DIM), generator=_gen(seed, 40, dev), device=dev, dtype=torch.float32)
    q = q.to(torch.float8_e4m3fn).view(torch.uint8)
    weights = torch.randn((T, heads), generator=_gen(seed, 41, dev), device=dev, dtype=torch.float32) / 8.0
    cache = torch.empty((problem.num_pages, P * (INDEX_DIM + 4)), dtype=torch.uint8, device=dev)
    step = max(1, (1 << 26) // (P * INDEX_DIM))  # pages per draw (bounded memory)
    for p0 in range(0, problem.num_pages, step):
        n = min(step, problem.num_pages - p0)
        g = _gen(seed, 2000 + p0 // step, dev)
        k = torch.randn((n, P * INDEX_DIM), generator=g, device=dev, dtype=torch.float32) * 32.0
        cache[p0:p0 + n, :P * INDEX_DIM] = k.to(torch.float8_e4m3fn).view(torch.uint8)
        e = torch.randint(-10, -3, (n, P), generator=g, device=dev).to(torch.float32)
        cache[p0:p0 + n, P * INDEX_DIM:] = torch.exp2(e).contiguous().view(torch.uint8).view(n, P * 4)
    return IndexerInputs(q=q, weights=weights, cache=cache, ctx=problem.ctx.to(torch.int32).to(dev), heads=heads)


# ------------------------------------------------------------------------------ fused-store inputs


@dataclasses.dataclass
class StoreInputs:
    """Inputs of the cache write fused with the latent's RMSNorm and the RoPE rotation.

    latent [n, 512] and rope [n, 64] bf16 (N(0, 1) * 3 and N(0, 1)), weight [512] bf16
    (1 + N(0, 1) / 10), positions [n] int64 uniform in [0, max_position), cos_sin
    [max_position, 64] fp32: cos, then sin, of position * 10000^(-j / 32) for the 32 pairs
    (the rotary table a model passes in; drawn here, not computed by the method).
    """

    latent: torch.Tensor
    rope: torch.Tensor
    weight: torch.Tensor
    positions: torch.Tensor
    cos_sin: torch.Tensor


def make_store_inputs(n: int, seed: int, max_position: int = 4096, device="cpu") -> StoreInputs:
    g = _gen(seed, 60, "cpu")
    latent = (torch.randn((n, LATENT_DIM), generator=g) * 3.0).to(torch.bfloat16)
    rope = torch.randn((n, ROPE_DIM), generator=g).to(torch.bfloat16)
    weight = (1.0 + torch.randn((LATENT_DIM,), generator=g) / 10.0).to(torch.bfloat16)
    positions = torch.randint(0, max_position, (n,), generator=g, dtype=torch.int64)
    theta = torch.pow(10000.0, -torch.arange(ROPE_DIM // 2, dtype=torch.float64) / (ROPE_DIM // 2))
    ang = torch.arange(max_position, dtype=torch.float64)[:, None] * theta[None, :]
    cos_sin = torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).to(torch.float32)
    d = torch.device(device)
    return StoreInputs(latent.to(d), rope.to(d), weight.to(d), positions.to(d), cos_sin.to(d))


def make_topk_variants(problem: Problem, n: int) -> list[torch.Tensor]:
    """n further index sets of a problem [T, K] int32 (same contexts, pages and padding recipe as
    its own: distinct request-local slots drawn uniformly from each token's visible prefix, in
    random order, -1 tail), each from its own seeded generator: consecutive end-to-end steps
    then gather different rows."""
    w = problem.w
    T, K = w.num_tokens, w.topk
    out = []
    for v in range(n):
        g = _gen(problem.seed, 300 + v, problem.device)
        topk = torch.full((T, K), -1, dtype=torch.int32)
        for t in range(T):
            r, i = divmod(t, w.next_n)
            visible = int(problem.ctx[r]) - (w.next_n - 1) + i
            nvalid = min(visible, K - w.tail_pad)
            idx = torch.randperm(visible, generator=g, device=problem.device)[:nvalid]
            topk[t, :nvalid] = idx.to(torch.int32).cpu()
        out.append(topk)
    return out
