"""The five synthetic decode-attention workloads and their seeded inputs.

Shapes follow the model shapes the pages use (Llama-3.1-8B: 32 layers,
32 query heads, 8 KV heads, d_h 128; Llama-3-70B: 80 layers, 64 query
heads, 8 KV heads) and the 16-token block of a vLLM-style paged cache.
Each workload describes only inputs and their structure: which physical
blocks a request owns, its context length, which token slots are evicted,
and the seeded q/K/V values.  No attention arithmetic lives here.

Generated tensors are bf16 (values drawn in float32, rounded to nearest
even).  Per-element randomness comes from ``gen`` so that a CPU call and a
CUDA call return identical bits.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

from . import gen


@dataclass
class Workload:
    name: str
    L: int
    n_q: int
    n_kv: int
    d_h: int
    batch: int
    kv_dtype: str                       # "bf16", "fp8_e4m3", "mixed" (a format per physical block),
                                        # "int4" or "int2" (codes with a scale and zero per group),
                                        # "angle" (angle-domain keys, FP8 values)
    block_size: int = 16
    seed: int = 0
    steps: int = 1                      # decode steps in one unit of work
    key_scale_range: tuple | None = None   # per-(layer, kv head) K factor ~ U[lo, hi]
    outlier_p: float = 0.0              # per-(layer, kv head, channel) outlier probability
    outlier_factor: float = 1.0
    evict_frac: float = 0.0             # fraction of unprotected slots evicted
    protect_prompt: int = 0             # leading tokens never evicted (prompt, sinks)
    protect_recent: int = 0             # trailing tokens never evicted
    scores: bool = False                # accumulate the importance score s_i
    pool_slack_blocks: int = 0          # unused physical blocks added to the pool
    mixed_probs: tuple | None = None    # mixed pools: P(BF16), P(E4M3), P(E5M2) of a physical block
    group_size: int = 0                 # low-bit pools: values per scale group (32, 64 or 128)
    description: str = ""
    _ctx0: list = field(default_factory=list)   # context before step 0's append

    # ------------------------------------------------------------------ shape
    @property
    def g(self) -> int:
        return self.n_q // self.n_kv

    @property
    def w_kv(self) -> float:
        """Bytes per stored K or V element (a single-format pool)."""
        if self.kv_dtype == "mixed":
            raise ValueError("a mixed pool has a w_kv per block: use token_bytes()")
        return {"bf16": 2, "fp8_e4m3": 1, "int4": 0.5, "int2": 0.25, "angle": 1}[self.kv_dtype]

    @property
    def lowbit(self) -> tuple | None:
        """(bits, group_size) of a low-bit pool, else None."""
        if self.kv_dtype in ("int4", "int2"):
            return (4 if self.kv_dtype == "int4" else 2, self.group_size)
        return None

    def seq_lens(self, step: int = 0) -> list[int]:
        """Attended context of every sequence at ``step`` (includes the token appended in it)."""
        if self.steps > 1:
            return [c + step + 1 for c in self._ctx0]
        return list(self._ctx0)

    def max_ctx(self) -> int:
        return max(self.seq_lens(self.steps - 1))

    def blocks_per_seq(self) -> list[int]:
        last = self.seq_lens(self.steps - 1)
        return [-(-c // self.block_size) for c in last]

    def max_blocks(self) -> int:
        return max(self.blocks_per_seq())

    def num_blocks(self) -> int:
        return sum(self.blocks_per_seq()) + self.pool_slack_blocks

    def append_pos(self, step: int = 0) -> list[int]:
        """Position written by the decode-step append of ``step``, per sequence."""
        return [c - 1 for c in self.seq_lens(step)]

    def _tokens_by_width(self, step: int = 0) -> tuple[int, int]:
        """(tokens attended in 2-byte storage, tokens in 1-byte storage) at ``step``."""
        tokens = sum(self.seq_lens(step))
        if self.kv_dtype != "mixed":
            return (tokens, 0) if self.kv_dtype == "bf16" else (0, tokens)   # angle: FP8-sized records
        fmt = self.block_formats()
        bt = self.block_table()
        wide = 0
        for b, n in enumerate(self.seq_lens(step)):
            full, tail = divmod(n, self.block_size)
            ids = bt[b, :full].numpy()
            wide += int((fmt[ids] == 0).sum()) * self.block_size
            if tail and fmt[int(bt[b, full])] == 0:
                wide += tail
        return wide, tokens - wide

    def kv_bytes_per_step(self, step: int = 0) -> int:
        """Closed-form K/V bytes attended in one step over all layers: 2·L·n_kv·d_h·w_kv per token
        (w_kv of the block that holds the token in a mixed pool)."""
        if self.lowbit:
            return 2 * self.L * self.n_kv * self.d_h * self.lowbit[0] * sum(self.seq_lens(step)) // 8
        wide, narrow = self._tokens_by_width(step)
        return 2 * self.L * self.n_kv * self.d_h * (2 * wide + narrow)

    def scale_bytes_per_step(self, step: int = 0) -> int:
        """Scale bytes read with the tokens: 8-bit tokens one fp32 scale for K and one for V per
        (token, KV head); low-bit tokens a half-precision scale and zero point per group, for K
        and for V."""
        if self.lowbit:
            return 2 * self.L * self.n_kv * 4 * (self.d_h // self.group_size) * sum(self.seq_lens(step))
        return 2 * self.L * self.n_kv * 4 * self._tokens_by_width(step)[1]

    def block_formats(self):
        """Mixed pools: uint8 numpy [num_blocks], the storage format of every physical block
        (0 BF16, 1 E4M3, 2 E5M2), drawn per block with probabilities mixed_probs."""
        import numpy as np

        p = self.mixed_probs or (1.0, 0.0, 0.0)
        u = gen.uniform(gen.stream_key(self.seed, self.name, "fmt"), gen.index_range(0, self.num_blocks(), "cpu"))
        u = u.double().numpy()
        return np.where(u < p[0], 0, np.where(u < p[0] + p[1], 1, 2)).astype(np.uint8)

    # ------------------------------------------------------------- structure
    def block_table(self) -> torch.Tensor:
        """int32 [batch][max_blocks]; logical block j of request b -> physical block (-1 = unused)."""
        nb = self.num_blocks()
        perm = gen.permutation(gen.stream_key(self.seed, self.name, "perm"), nb)
        bt = torch.full((self.batch, self.max_blocks()), -1, dtype=torch.int32)
        off = 0
        for b, n in enumerate(self.blocks_per_seq()):
            bt[b, :n] = perm[off:off + n].to(torch.int32)
            off += n
        return bt

    def evicted_positions(self, b: int) -> torch.Tensor:
        """Sorted logical positions of request b whose slots are evicted (fixed over all steps)."""
        if self.evict_frac <= 0:
            return torch.zeros(0, dtype=torch.int64)
        lo = self.protect_prompt
        hi = self._ctx0[b] - self.protect_recent
        n = hi - lo
        if n <= 0:                       # a context shorter than its protected parts: nothing evictable
            return torch.zeros(0, dtype=torch.int64)
        k = int(round(self.evict_frac * n))
        pick = gen.choose(gen.stream_key(self.seed, self.name, "evict", b), n, k)
        return pick + lo

    def retain_mask(self, block_table: torch.Tensor | None = None) -> torch.Tensor | None:
        """uint16-valued int32 [num_blocks]: bit o set = slot o of that physical block is kept."""
        if self.evict_frac <= 0:
            return None
        bt = self.block_table() if block_table is None else block_table
        mask = torch.full((self.num_blocks(),), 0xFFFF, dtype=torch.int32)
        for b in range(self.batch):
            for pos in self.evicted_positions(b).tolist():
                p = int(bt[b, pos // self.block_size])
                mask[p] &= ~(1 << (pos % self.block_size)) & 0xFFFF
        return mask

    def slot_mapping(self, b: int, pos0: int, pos1: int, block_table: torch.Tensor) -> torch.Tensor:
        """int64 pool slot (physical block · block_size + offset) of positions [pos0, pos1) of request b."""
        pos = torch.arange(pos0, pos1, dtype=torch.int64)
        blk = block_table[b].to(torch.int64)[pos // self.block_size]
        return blk * self.block_size + pos % self.block_size

    # ----------------------------------------------------------------- values
    def _key_factor(self, layer: int, device) -> torch.Tensor:
        """float32 [n_kv]: per-(layer, kv head) multiplier of K."""
        if self.key_scale_range is None:
            return torch.ones(self.n_kv, dtype=torch.float32, device=device)
        lo, hi = self.key_scale_range
        u = gen.uniform(gen.stream_key(self.seed, self.name, "kscale", layer),
                        gen.index_range(0, self.n_kv, device))
        return (torch.tensor(lo, dtype=torch.float32, device=device)
                + u * torch.tensor(hi - lo, dtype=torch.float32, device=device))

    def _outlier_factor(self, layer: int, which: str, device) -> torch.Tensor:
        """float32 [n_kv][d_h]: outlier_factor on outlier channels, 1 elsewhere."""
        ones = torch.ones(self.n_kv, self.d_h, dtype=torch.float32, device=device)
        if self.outlier_p <= 0:
            return ones
        u = gen.uniform(gen.stream_key(self.seed, self.name, "outlier", which, layer),
                        gen.index_range(0, self.n_kv * self.d_h, device)).view(self.n_kv, self.d_h)
        f = torch.tensor(self.outlier_factor, dtype=torch.float32, device=device)
        return torch.where(u < self.outlier_p, f, ones)

    def q(self, layer: int, step: int = 0, device="cpu") -> torch.Tensor:
        """bf16 [batch][n_q][d_h] query of ``layer`` at ``step``, ~N(0, 1)."""
        n = self.batch * self.n_q * self.d_h
        x = gen.normal(gen.stream_key(self.seed, self.name, "q", layer, step), gen.index_range(0, n, device))
        return x.view(self.batch, self.n_q, self.d_h).to(torch.bfloat16)

    def kv(self, layer: int, b: int, pos0: int, pos1: int, device="cpu"):
        """bf16 (K, V), each [pos1 - pos0][n_kv][d_h], of positions [pos0, pos1) of request b."""
        per = self.n_kv * self.d_h
        idx = gen.index_range(pos0 * per, (pos1 - pos0) * per, device)
        shape = (pos1 - pos0, self.n_kv, self.d_h)
        k = gen.normal(gen.stream_key(self.seed, self.name, "k", layer, b), idx).view(shape)
        v = gen.normal(gen.stream_key(self.seed, self.name, "v", layer, b), idx).view(shape)
        k = k * self._key_factor(layer, device).view(1, self.n_kv, 1)
        k = k * self._outlier_factor(layer, "k", device).unsqueeze(0)
        v = v * self._outlier_factor(layer, "v", device).unsqueeze(0)
        return k.to(torch.bfloat16), v.to(torch.bfloat16)


def _log_uniform_lens(seed: int, name: str, n: int, lo: int, hi: int) -> list[int]:
    u = gen.uniform(gen.stream_key(seed, name, "ctx"), gen.index_range(0, n, "cpu")).double().tolist()
    a, b = math.log(lo), math.log(hi)
    return [max(lo, min(hi, int(math.exp(a + x * (b - a))))) for x in u]


def tiny(seed: int = 0) -> Workload:
    w = Workload("tiny", L=1, n_q=32, n_kv=8, d_h=128, batch=1, kv_dtype="bf16", seed=seed,
                 pool_slack_blocks=128,
                 description="1 layer, batch 1, n_q 32, n_kv 8, d_h 128, context 2,048, "
                             "128 blocks in a shuffled pool of 256, bf16 KV")
    w._ctx0 = [2048]
    return w


def llama8b(seed: int = 0) -> Workload:
    w = Workload("llama8b", L=32, n_q=32, n_kv=8, d_h=128, batch=32, kv_dtype="bf16", seed=seed,
                 key_scale_range=(0.5, 2.0),
                 description="Llama-3.1-8B shape decode step: 32 layers, n_q 32, n_kv 8, d_h 128, "
                             "batch 32, context 8,192, bf16 KV, 16,384-block pool per layer")
    w._ctx0 = [8192] * 32
    return w


def llama8b_mixed(seed: int = 0) -> Workload:
    w = Workload("llama8b_mixed", L=32, n_q=32, n_kv=8, d_h=128, batch=32, kv_dtype="mixed", seed=seed,
                 key_scale_range=(0.5, 2.0), mixed_probs=(0.25, 0.5, 0.25),
                 description="Llama-3.1-8B shape decode step, mixed-precision pages: 32 layers, n_q 32, n_kv 8, "
                             "d_h 128, batch 32, context 8,192, each physical block BF16 / FP8-E4M3 / FP8-E5M2 "
                             "with probability 1/4, 1/2, 1/4")
    w._ctx0 = [8192] * 32
    return w


def ragged(seed: int = 0) -> Workload:
    w = Workload("ragged", L=4, n_q=32, n_kv=8, d_h=128, batch=64, kv_dtype="bf16", seed=seed,
                 description="8B shape, 4 layers, 64 requests, context log-uniform in [256, 32,768], bf16 KV")
    w._ctx0 = _log_uniform_lens(seed, w.name, 64, 256, 32768)
    return w


def llama70b_fp8(seed: int = 0) -> Workload:
    w = Workload("llama70b_fp8", L=80, n_q=64, n_kv=8, d_h=128, batch=1, kv_dtype="fp8_e4m3", seed=seed,
                 outlier_p=0.001, outlier_factor=20.0,
                 description="Llama-3-70B shape long context: 80 layers, n_q 64, n_kv 8, d_h 128, batch 1, "
                             "context 131,072, FP8-e4m3 KV with per-(token, head) scale, 0.1% outlier channels x20")
    w._ctx0 = [131072]
    return w


def tiered(seed: int = 0) -> Workload:
    w = Workload("tiered", L=28, n_q=28, n_kv=4, d_h=128, batch=8, kv_dtype="bf16", seed=seed,
                 steps=64, evict_frac=0.03, protect_prompt=512, protect_recent=256, scores=True,
                 description="reasoning-trace cache: 28 layers, n_q 28, n_kv 4, d_h 128, batch 8, "
                             "context 16,384 growing over 64 steps, 3% of unprotected slots evicted, "
                             "importance scores accumulated")
    w._ctx0 = [16384] * 8
    return w


def llama70b_int4(seed: int = 0) -> Workload:
    w = Workload("llama70b_int4", L=80, n_q=64, n_kv=8, d_h=128, batch=1, kv_dtype="int4", seed=seed,
                 outlier_p=0.001, outlier_factor=20.0, group_size=32,
                 description="Llama-3-70B shape long context, 4-bit KV: 80 layers, n_q 64, n_kv 8, d_h 128, batch 1, "
                             "context 131,072, 4-bit codes with a half-precision scale and zero point per group of "
                             "32 values, 0.1% outlier channels x20")
    w._ctx0 = [131072]
    return w


def llama70b_int2(seed: int = 0) -> Workload:
    w = Workload("llama70b_int2", L=80, n_q=64, n_kv=8, d_h=128, batch=1, kv_dtype="int2", seed=seed,
                 outlier_p=0.001, outlier_factor=20.0, group_size=32,
                 description="Llama-3-70B shape long context, 2-bit KV: 80 layers, n_q 64, n_kv 8, d_h 128, batch 1, "
                             "context 131,072, 2-bit codes with a half-precision scale and zero point per group of "
                             "32 values, 0.1% outlier channels x20")
    w._ctx0 = [131072]
    return w


def llama70b_angle(seed: int = 0) -> Workload:
    w = Workload("llama70b_angle", L=80, n_q=64, n_kv=8, d_h=128, batch=1, kv_dtype="angle", seed=seed,
                 outlier_p=0.001, outlier_factor=20.0,
                 description="Llama-3-70B shape long context, angle-domain keys: 80 layers, n_q 64, n_kv 8, d_h 128, "
                             "batch 1, context 131,072, keys as an FP8-e4m3 direction code plus a radius factor per "
                             "(token, head), FP8-e4m3 values, 0.1% outlier channels x20")
    w._ctx0 = [131072]
    return w


WORKLOADS = {"tiny": tiny, "llama8b": llama8b, "llama8b_mixed": llama8b_mixed, "ragged": ragged,
             "llama70b_fp8": llama70b_fp8, "tiered": tiered, "llama70b_int4": llama70b_int4,
             "llama70b_int2": llama70b_int2, "llama70b_angle": llama70b_angle}


def get(name: str, seed: int = 0) -> Workload:
    return WORKLOADS[name](seed)
