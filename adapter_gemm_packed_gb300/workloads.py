"""Seeded synthetic inputs for the packed multi-adapter LoRA layer.

This module draws the numbers both sides of every parity check consume: the
CUDA path (through the C-ABI binding) and the fp64 CPU oracle.  It holds none
of the layer's arithmetic: it only samples shapes, ranks, token counts and
Gaussian tensors, rounds the activation/weight tensors to bfloat16 where the
workload says so, and hands back plain numpy arrays in the storage layout the
library uses:

  * ``Wt``  = W transposed, ``[d_out, d_in]`` (the frozen base weight),
  * ``At[i]`` = A_i transposed, ``[r_i, d_in]`` (fp32 master),
  * ``Bt[i]`` = B_i transposed, ``[d_out, r_i]`` (fp32 master),
  * ``X`` ``[N, d_in]`` and ``dY`` ``[N, d_out]``, the packed token rows, job i
    owning rows ``[offset_i, offset_i + n_i)``.

bf16 tensors are returned as ``uint16`` bit patterns (round-to-nearest-even
from the fp32 draw); fp32 tensors as ``float32``.

Randomness: every tensor has its own counter-based Philox stream keyed by
``(config_id, tensor_id, chunk)``, drawn in fixed chunks of ``CHUNK`` elements,
so a tensor's values do not depend on how many threads draw it nor on which
other tensors were drawn before it.  Init distributions follow the workload
descriptions (PLoRA, §2.1 for the LoRA shapes; §4.1/§11.2.1 for the model
dimensions): ``N(0, 1/d_in)`` is a variance, ``N(0, 0.02)`` a standard deviation.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field

import numpy as np

CHUNK = 1 << 22

# tensor ids inside one config's key space
T_RANKS, T_TOKENS, T_W, T_X, T_DY, T_MISC = 0, 1, 2, 3, 4, 5
T_ADAPTER_BASE = 100          # A_i -> 100 + 4 i, B_i -> 101 + 4 i, extras 102/103 + 4 i


def _key(cfg_id: int, tensor_id: int, chunk: int) -> np.ndarray:
    return np.array([cfg_id & 0xFFFFFFFFFFFFFFFF, ((tensor_id & 0xFFFFFFFF) << 32) | (chunk & 0xFFFFFFFF)],
                    dtype=np.uint64)


def rng(cfg_id: int, tensor_id: int, chunk: int = 0) -> np.random.Generator:
    """Counter-based generator for one chunk of one tensor."""
    return np.random.Generator(np.random.Philox(key=_key(cfg_id, tensor_id, chunk)))


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal_f32(cfg_id: int, tensor_id: int, n: int, std: float) -> np.ndarray:
    """``n`` fp32 draws of N(0, std^2), chunked so the values are thread-count independent."""
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK

    def work(c: int) -> None:
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        seg = out[lo:hi]
        rng(cfg_id, tensor_id, c).standard_normal(out=seg, dtype=np.float32)
        if std != 1.0:
            seg *= np.float32(std)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with _cf.ThreadPoolExecutor(min(_threads(), nchunks)) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def normal_range(cfg_id: int, tensor_id: int, lo: int, hi: int, std: float, bf16: bool = False) -> np.ndarray:
    """Elements [lo, hi) of the tensor that ``normal_f32(cfg_id, tensor_id, n, std)`` draws (for any
    n >= hi), drawing only the chunks that hold them; rounded to bf16 bit patterns if ``bf16``.
    The values are those of the whole-tensor draw, element for element."""
    out = np.empty(max(0, hi - lo), dtype=np.uint16 if bf16 else np.float32)
    if hi <= lo:
        return out
    c0, c1 = lo // CHUNK, (hi - 1) // CHUNK + 1

    def work(c: int) -> None:
        a, b = max(lo, c * CHUNK), min(hi, (c + 1) * CHUNK)
        seg = np.empty(min(b, (c + 1) * CHUNK) - c * CHUNK, dtype=np.float32)
        rng(cfg_id, tensor_id, c).standard_normal(out=seg, dtype=np.float32)
        part = seg[a - c * CHUNK:]
        if std != 1.0:
            part *= np.float32(std)
        out[a - lo:b - lo] = to_bf16_bits(part) if bf16 else part

    if c1 - c0 <= 1:
        work(c0)
    else:
        with _cf.ThreadPoolExecutor(min(_threads(), c1 - c0)) as ex:
            list(ex.map(work, range(c0, c1)))
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bfloat16 (round to nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to fp32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Workload:
    """Sizes and seeds of one packed LoRA layer problem (no tensors)."""
    name: str
    cfg_id: int
    d_in: int
    d_out: int
    dtype: str                       # "f32" or "bf16": dtype of X, W, dY, Y, dX
    ranks: list
    n_tokens: list
    alphas: list
    w_std: float
    a_std: float
    b_std: float
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    # Shared-input pack: output widths of the projections stacked in W (None = one projection).
    # Then ``ranks`` / ``alphas`` hold one entry per (job, projection), job-major, and adapter
    # entry i = j * G + g has Bt [groups[g], r].
    groups: list = None

    @property
    def n_adapters(self) -> int:
        return len(self.ranks)

    @property
    def n_groups(self) -> int:
        return 1 if self.groups is None else len(self.groups)

    @property
    def widths(self) -> list:
        return [self.d_out] if self.groups is None else list(self.groups)

    @property
    def group_offsets(self) -> list:
        w = self.widths
        return [sum(w[:g]) for g in range(len(w))]

    @property
    def entry_tokens(self) -> list:
        """Tokens of each adapter entry (a job's count repeated once per projection)."""
        return [n for n in self.n_tokens for _ in range(self.n_groups)]

    @property
    def entry_width(self) -> list:
        """Output width of each adapter entry's B."""
        return [w for _ in self.n_tokens for w in self.widths]

    def nest(self, flat) -> list:
        """Per-entry list -> per-job lists of per-projection values."""
        G = self.n_groups
        return [list(flat[j * G:(j + 1) * G]) for j in range(len(self.n_tokens))]

    @property
    def offsets(self) -> list:
        off, out = 0, []
        for n in self.n_tokens:
            out.append(off)
            off += n
        return out

    @property
    def N(self) -> int:
        return int(sum(self.n_tokens))


@dataclass
class Tensors:
    """Materialised inputs of a :class:`Workload` (numpy, storage layout)."""
    wl: Workload
    Wt: np.ndarray
    X: np.ndarray
    dY: np.ndarray
    At: list = field(default_factory=list)
    Bt: list = field(default_factory=list)


# --------------------------------------------------------------------------
# The five workloads (sizes from the packed-LoRA pages' model shapes; see
# PLoRA §4.1 for the Llama-3/Qwen dimensions and §11.2.1 for the microbench
# ranges).  Unstated alphas follow the tiny config (alpha = 2 r).
# --------------------------------------------------------------------------

def tiny_f32() -> Workload:
    """d=256, ranks {4,8,16}, segments {64,32,96}, alpha=2r, fp32."""
    d = 256
    return Workload("tiny_f32_d256_r4-8-16", 1, d, d, "f32", [4, 8, 16], [64, 32, 96],
                    [8.0, 16.0, 32.0], w_std=(1.0 / d) ** 0.5, a_std=(1.0 / d) ** 0.5, b_std=0.02)


def llama8b_qproj() -> Workload:
    """q_proj 4096x4096 bf16, 8 adapters ranks {8,8,16,16,32,32,64,64}, 2048 tokens each."""
    ranks = [8, 8, 16, 16, 32, 32, 64, 64]
    return Workload("llama3_8b_q_proj_4096x4096_8ad_16384tok", 2, 4096, 4096, "bf16", ranks, [2048] * 8,
                    [2.0 * r for r in ranks], w_std=0.02, a_std=(1.0 / 4096) ** 0.5, b_std=0.02)


def llama8b_qproj_tiny_ranks() -> Workload:
    """The q_proj shape and tokens with ranks {1,1,2,2,4,4,4,4}: the small-rank regime, where the
    shrink, dH, dA and dB are matrix-vector-like products (r FLOP per byte of X or dY)."""
    ranks = [1, 1, 2, 2, 4, 4, 4, 4]
    return Workload("llama3_8b_q_proj_4096x4096_8ad_16384tok_r1-4", 53, 4096, 4096, "bf16", ranks, [2048] * 8,
                    [2.0 * r for r in ranks], w_std=0.02, a_std=(1.0 / 4096) ** 0.5, b_std=0.02)


def llama8b_qproj_f32() -> Workload:
    """The q_proj workload with fp32 activations and weight (the true-fp32 FFMA path at a real size)."""
    q = llama8b_qproj()
    return Workload("llama3_8b_q_proj_4096x4096_8ad_16384tok_f32", 55, 4096, 4096, "f32", q.ranks, q.n_tokens,
                    q.alphas, w_std=0.02, a_std=(1.0 / 4096) ** 0.5, b_std=0.02)


def mlp_up_lognormal() -> Workload:
    """4096->14336 bf16, 16 adapters, ranks U{4..128}, tokens lognormal(7,1) rounded to 16, clipped [64,8192], alpha=16."""
    cfg = 3
    g = rng(cfg, T_RANKS)
    ranks = [int(r) for r in g.choice(np.array([4, 8, 16, 32, 64, 128]), size=16)]
    g = rng(cfg, T_TOKENS)
    raw = g.lognormal(mean=7.0, sigma=1.0, size=16)
    toks = [int(min(8192, max(64, int(np.rint(v / 16.0)) * 16))) for v in raw]
    return Workload("mlp_up_4096x14336_16ad_lognormal", cfg, 4096, 14336, "bf16", ranks, toks,
                    [16.0] * 16, w_std=0.02, a_std=(1.0 / 4096) ** 0.5, b_std=0.02)


LLAMA8B_PROJ = [("q", 4096, 4096), ("k", 4096, 1024), ("v", 4096, 1024), ("o", 4096, 4096),
                ("gate", 4096, 14336), ("up", 4096, 14336), ("down", 14336, 4096)]


def llama8b_layer(proj: int) -> Workload:
    """One of the 7 projections of a Llama-3-8B decoder layer, 32 adapters, seq 1024, 1..8 seqs per job."""
    cfg = 4
    g = rng(cfg, T_RANKS)
    ranks = [int(r) for r in g.choice(np.array([8, 16, 32, 64, 128]), size=32)]
    g = rng(cfg, T_TOKENS)
    toks = [int(b) * 1024 for b in g.integers(1, 9, size=32)]
    name, din, dout = LLAMA8B_PROJ[proj]
    return Workload(f"llama3_8b_layer_{name}_{din}x{dout}_32ad", 40 + proj, din, dout, "bf16", ranks, toks,
                    [2.0 * r for r in ranks], w_std=0.02, a_std=(1.0 / 4096) ** 0.5, b_std=0.02)


def llama70b_down_many_small() -> Workload:
    """down_proj 28672->8192 bf16, 128 adapters, ranks {1..256} powers of two, segments 16..256 step 16, alpha=r."""
    cfg = 5
    g = rng(cfg, T_RANKS)
    ranks = [int(r) for r in g.choice(np.array([1 << k for k in range(9)]), size=128)]
    g = rng(cfg, T_TOKENS)
    toks = [int(v) * 16 for v in g.integers(1, 17, size=128)]
    return Workload("llama70b_down_28672x8192_128ad_small", cfg, 28672, 8192, "bf16", ranks, toks,
                    [float(r) for r in ranks], w_std=0.02, a_std=(1.0 / 4096) ** 0.5, b_std=0.02)


def llama70b_down_many_small_half() -> Workload:
    """The first 64 jobs of the many-small-jobs workload (same shape, ranks and token counts; own
    seeds): X 0.5 GB and dY 0.15 GB, still above the L2, about 4 GB on the device in all, a case
    small enough for detailed profiler captures."""
    full = llama70b_down_many_small()
    return custom(full.name + "_half", 56, full.d_in, full.d_out, full.ranks[:64], full.n_tokens[:64],
                  alphas=full.alphas[:64], a_std=full.a_std)


def custom(name: str, cfg_id: int, d_in: int, d_out: int, ranks, n_tokens, alphas=None, dtype="bf16",
           w_std=0.02, a_std=None, b_std=0.02) -> Workload:
    """Ad-hoc workload for edge-case tests (ragged tails, rank 1, straddling segments...)."""
    ranks = [int(r) for r in ranks]
    alphas = [2.0 * r for r in ranks] if alphas is None else [float(a) for a in alphas]
    a_std = (1.0 / d_in) ** 0.5 if a_std is None else a_std
    return Workload(name, cfg_id, d_in, d_out, dtype, ranks, [int(n) for n in n_tokens], alphas,
                    w_std=w_std, a_std=a_std, b_std=b_std)


def custom_grouped(name: str, cfg_id: int, d_in: int, widths, ranks_jg, n_tokens, alphas_jg=None, dtype="bf16",
                   w_std=0.02, a_std=None, b_std=0.02) -> Workload:
    """A shared-input pack: the projections of widths ``widths`` stacked in W, job j with rank
    ranks_jg[j][g] on projection g (alpha = 2 r unless given)."""
    ranks = [int(r) for rj in ranks_jg for r in rj]
    alphas = [2.0 * r for r in ranks] if alphas_jg is None else [float(a) for aj in alphas_jg for a in aj]
    a_std = (1.0 / d_in) ** 0.5 if a_std is None else a_std
    return Workload(name, cfg_id, d_in, int(sum(widths)), dtype, ranks, [int(n) for n in n_tokens], alphas,
                    w_std=w_std, a_std=a_std, b_std=b_std, groups=[int(w) for w in widths])


def llama8b_qkv_shared() -> Workload:
    """The q, k and v projections of a Llama-3-8B layer as one shared-input pack (4096 ->
    4096 + 1024 + 1024): the jobs, ranks and token counts of the per-projection layer workloads,
    each job's rank the same on all three projections."""
    q = llama8b_layer(0)
    ranks_jg = [[r, r, r] for r in q.ranks]
    wl = custom_grouped("llama3_8b_layer_qkv_shared_4096x6144_32ad", 50, 4096, [4096, 1024, 1024], ranks_jg,
                        q.n_tokens, a_std=(1.0 / 4096) ** 0.5)
    return wl


def llama8b_qkv_shared_small() -> Workload:
    """qkv_shared with an eighth of each job's tokens (about 18K; X and dY still above the L2),
    a case small enough for detailed profiler captures."""
    q = llama8b_layer(0)
    return custom_grouped("llama3_8b_layer_qkv_shared_4096x6144_32ad_eighth", 51, 4096, [4096, 1024, 1024],
                          [[r, r, r] for r in q.ranks], [n // 8 for n in q.n_tokens], a_std=(1.0 / 4096) ** 0.5)


def llama8b_layer_k_half() -> Workload:
    """The Llama-3-8B k projection workload with half of each job's tokens (about 72K; dY 147 MB, still
    above the L2), a case small enough for detailed profiler captures."""
    k = llama8b_layer(1)
    return custom("llama3_8b_layer_k_4096x1024_32ad_half", 54, 4096, 1024, k.ranks, [n // 2 for n in k.n_tokens],
                  alphas=k.alphas, a_std=(1.0 / 4096) ** 0.5)


def llama8b_qproj_w4() -> Workload:
    """The q_proj workload with a 4-bit base weight (int4 codes, fp32 scales per 64 inputs)."""
    wl = llama8b_qproj()
    wl.name = "llama3_8b_q_proj_4096x4096_8ad_16384tok_w4base"
    wl.cfg_id = 6
    wl.dtype = "bf16_w4"
    return wl


CONFIGS = {
    "tiny": tiny_f32,
    "qproj_w4": llama8b_qproj_w4,
    "qproj": llama8b_qproj,
    "qproj_tiny_ranks": llama8b_qproj_tiny_ranks,
    "qproj_f32": llama8b_qproj_f32,
    "mlp_up": mlp_up_lognormal,
    "many_small": llama70b_down_many_small,
    "many_small_half": llama70b_down_many_small_half,
    "qkv_shared": llama8b_qkv_shared,
    "qkv_shared_small": llama8b_qkv_shared_small,
    "k_proj_half": llama8b_layer_k_half,
}


def _act(wl: Workload, tid: int, n: int, std: float) -> np.ndarray:
    # bf16 tensors are rounded chunk by chunk in the drawing threads: the same values as
    # to_bf16_bits(normal_f32(...)), without the full-size fp32 intermediate
    return normal_range(wl.cfg_id, tid, 0, n, std, bf16=wl.dtype != "f32")


def _act_rows(wl: Workload, tid: int, width: int, rows, std: float) -> np.ndarray:
    """Rows ``rows`` (a list of (first, count) runs) of a [N, width] activation tensor."""
    parts = [normal_range(wl.cfg_id, tid, a * width, (a + k) * width, std, bf16=wl.dtype != "f32").reshape(k, width)
             for a, k in rows]
    return np.concatenate(parts) if parts else np.empty((0, width), np.uint16 if wl.dtype != "f32" else np.float32)


T_WQ, T_WSCALE = 6, 7


def w4_weight(wl: Workload):
    """A 4-bit base weight for a ``bf16_w4`` workload: uniformly random code bytes
    Wq [d_out, d_in/2] and positive fp32 group scales Wscale [d_in/64, d_out] around w_std/4,
    so the dequantised weight has about the spread of the bf16 workloads' W."""
    g = rng(wl.cfg_id, T_WQ)
    Wq = g.integers(0, 256, size=(wl.d_out, wl.d_in // 2), dtype=np.uint8)
    s = normal_f32(wl.cfg_id, T_WSCALE, (wl.d_in // 64) * wl.d_out, 0.1)
    Wscale = (np.float32(wl.w_std / 4.0) * (np.float32(1.0) + np.abs(s))).reshape(wl.d_in // 64, wl.d_out)
    return Wq, Wscale.astype(np.float32)


def materialise(wl: Workload, with_dY: bool = True) -> Tensors:
    """Draw every tensor of the workload (storage layout, see module doc).  For ``bf16_w4``
    workloads ``Wt`` is None and ``Wq`` / ``Wscale`` hold the 4-bit base."""
    N = wl.N
    if wl.dtype == "bf16_w4":
        Wt = None
    else:
        Wt = _act(wl, T_W, wl.d_out * wl.d_in, wl.w_std).reshape(wl.d_out, wl.d_in)
    X = _act(wl, T_X, N * wl.d_in, 1.0).reshape(N, wl.d_in)
    dY = _act(wl, T_DY, N * wl.d_out, 1.0).reshape(N, wl.d_out) if with_dY else None
    At, Bt = [], []
    for i, (r, w) in enumerate(zip(wl.ranks, wl.entry_width)):
        At.append(normal_f32(wl.cfg_id, T_ADAPTER_BASE + 4 * i, r * wl.d_in, wl.a_std).reshape(r, wl.d_in))
        Bt.append(normal_f32(wl.cfg_id, T_ADAPTER_BASE + 4 * i + 1, w * r, wl.b_std).reshape(w, r))
    T = Tensors(wl, Wt, X, dY, At, Bt)
    if wl.dtype == "bf16_w4":
        T.Wq, T.Wscale = w4_weight(wl)
    return T


def materialise_jobs(wl: Workload, jobs=None, per_job: int | None = None):
    """The pack made of jobs ``jobs`` of ``wl`` (indices, in that order; default all), each cut to
    its first ``per_job`` tokens if given, with the values ``materialise(wl)`` would give those
    rows and adapters.  Only the chunks holding the chosen rows are drawn.  Returns
    ``(sub, T)``: the sub-pack's Workload (same seeds, its own token table) and its Tensors.
    This is how a shard of a pack, or a bounded token sample of it, is built."""
    jobs = list(range(len(wl.n_tokens))) if jobs is None else [int(j) for j in jobs]
    G = wl.n_groups
    offs = wl.offsets
    toks = [wl.n_tokens[j] if per_job is None else min(per_job, wl.n_tokens[j]) for j in jobs]
    runs = [(offs[j], k) for j, k in zip(jobs, toks)]
    entries = [j * G + g for j in jobs for g in range(G)]
    sub = Workload(wl.name, wl.cfg_id, wl.d_in, wl.d_out, wl.dtype, [wl.ranks[i] for i in entries], toks,
                   [wl.alphas[i] for i in entries], wl.w_std, wl.a_std, wl.b_std, wl.lr, wl.beta1, wl.beta2, wl.eps,
                   wl.weight_decay, None if wl.groups is None else list(wl.groups))
    if wl.dtype == "bf16_w4":
        Wt = None
    else:
        Wt = _act(wl, T_W, wl.d_out * wl.d_in, wl.w_std).reshape(wl.d_out, wl.d_in)
    X = _act_rows(wl, T_X, wl.d_in, runs, 1.0)
    dY = _act_rows(wl, T_DY, wl.d_out, runs, 1.0)
    width = wl.entry_width
    At = [normal_f32(wl.cfg_id, T_ADAPTER_BASE + 4 * i, wl.ranks[i] * wl.d_in, wl.a_std).reshape(wl.ranks[i], wl.d_in)
          for i in entries]
    Bt = [normal_f32(wl.cfg_id, T_ADAPTER_BASE + 4 * i + 1, width[i] * wl.ranks[i], wl.b_std)
          .reshape(width[i], wl.ranks[i]) for i in entries]
    T = Tensors(sub, Wt, X, dY, At, Bt)
    if wl.dtype == "bf16_w4":
        T.Wq, T.Wscale = w4_weight(wl)
    return sub, T


@dataclass
class Layer:
    """Several projections trained as one step (a decoder layer): each part is a Workload with
    its own base weight, inputs and adapters; all parts share the job table (token counts and
    ranks), so the layer's tokens per step are one part's N."""
    name: str
    parts: list

    @property
    def N(self) -> int:
        return self.parts[0].N

    @property
    def n_tokens(self) -> list:
        return self.parts[0].n_tokens

    @property
    def ranks(self) -> list:
        return self.parts[0].ranks


def llama8b_layer_all(token_div: int = 1) -> Layer:
    """All seven projections of a Llama-3-8B decoder layer (q, k, v, o, gate, up, down) with the
    32 jobs of the per-projection layer workloads: every job has the same rank and tokens on each
    projection, and each projection its own X, dY and adapters.  ``token_div`` > 1 keeps
    1/token_div of every job's tokens (own seeds), a smaller case of the same layer."""
    parts = [llama8b_layer(p) for p in range(len(LLAMA8B_PROJ))]
    if token_div != 1:
        parts = [custom(f"{w.name}_div{token_div}", 60 + 8 * token_div + p, w.d_in, w.d_out, w.ranks,
                        [n // token_div for n in w.n_tokens], alphas=w.alphas, a_std=w.a_std)
                 for p, w in enumerate(parts)]
    return Layer(f"llama3_8b_layer_7proj_32ad_{parts[0].N}tok", parts)


def optimizer_state(wl: Workload, which: str, i: int, shape, kind: str) -> np.ndarray:
    """Seeded fp32 stand-ins for a gradient (``kind='g'``), a first moment (``'m'``) or a
    second moment (``'v'``, non-negative) of adapter ``i``'s ``which`` in {'A','B'}."""
    n = int(np.prod(shape))
    tid = 10_000 + 8 * i + (0 if which == "A" else 4) + {"g": 0, "m": 1, "v": 2}[kind]
    x = normal_f32(wl.cfg_id, tid, n, 1e-2 if kind != "v" else 1e-2)
    if kind == "v":
        x = x * x
    return x.reshape(shape)


def rows_as_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 view of stored values (bf16 bit patterns or fp32)."""
    if dtype in ("bf16", "bf16_w4"):
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float64)
