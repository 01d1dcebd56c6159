"""Benchmark: paged GQA decode attention steps on GB300 through the C ABI.

One step = one decode step of every layer of the workload: per layer one
kvd_decode_attn call: the decode kernel appends the new token's K/V of every request and
runs paged decode attention with split-KV; a second launch merges the splits.  The tiered
workload adds each layer's share of the importance score (a score launch on a second
stream, or --fused-scores: inside the merge launch).  Layers run in order, as
in a model where layer ℓ+1's query depends on layer ℓ.  The L-layer step is captured as a
CUDA graph and replayed.

Prints one JSON line.  `value` is the closed-form K/V bytes attended per step,
2·L·n_kv·d_h·w_kv per token (FP8 scales excluded), divided by the step time, in GB/s,
with every input resident in HBM.  Default workload: Llama-3.1-8B shape, 32 layers,
batch 32, context 8,192, BF16 KV (34.4 GB of KV per step, far larger than L2).  The
default run also times the ragged, 70B FP8, tiered, mixed-precision, 70B INT4 / 2-bit and
70B angle-domain workloads (key `workloads`, each with its own value, roofline and clocks), and measures the
read-only HBM stream (`hbm_read_peak`) beside the copy peak of MEASURED_PEAKS.json.  For the
8-bit and low-bit pools the roofline counts the scales (and zero points) with the codes.

`--impl reference` times the fp64 CPU oracle instead: each step is a bounded sample of the
workload, one whole (layer, request) unit per host thread.

Host tier (T1): `--host-tier F` moves the fraction F of each request's least important
unprotected blocks to pinned host memory before timing; the decode kernel reads them in
place over the host link (`--host-tier-staged`: copied per layer into HBM by a DMA on a
copy stream instead).  `--retier` (tiered workload) reassigns tiers from the live
importance scores every 64 steps inside the timed loop.  The K/V bytes counted per step
are the same as without a tier; `launch.host_tier` reports the host-tier bytes per step and
the costs of the plan and the moves.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn KV HBM GB/s and % of GB300 HBM peak; attention steps/s"
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- analytic
def kv_bytes_per_token(L: int, n_kv: int, d_h: int, w_kv: float) -> float:
    """2·L·n_kv·d_h·w_kv: K and V of every layer and KV head."""
    return 2 * L * n_kv * d_h * w_kv


def traffic_crossover_tokens(params: float, w_p: float, batch: int, per_token: float) -> float:
    """Context s* where per-step KV bytes b·s·per_token equal the weight bytes P·w_p."""
    return params * w_p / (batch * per_token)


def kv_speedup(weight_bytes: float, kv_bytes: float, c: float) -> float:
    """Memory-bound step-time ratio when the KV bytes shrink by c: (W + KV) / (W + KV/c)."""
    return (weight_bytes + kv_bytes) / (weight_bytes + kv_bytes / c)


def decode_intensity(g: int, w_kv: float) -> float:
    """Long-context FLOP per KV byte of GQA decode: 2 FLOP per (q, k) and (p, v) element, g heads."""
    return 2 * g / w_kv


DECODE_SOURCES = ("kvd_decode.cu", "kvd_common.cuh", "kvd_internal.h", "kvd_decode_kernel.cuh", "kvd_decode_lowbit.cu")


def decode_source_digest():
    """sha256 of the decode kernel's sources (DECODE_SOURCES concatenated in that order), or None if
    one is missing."""
    import hashlib

    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        src = os.path.join(ROOT, "paged_gqa_decode_kvd_gb300", "csrc", name)
        if not os.path.exists(src):
            return None
        h.update(open(src, "rb").read())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on the
    current decode kernel sources (matched by decode_source_digest); otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    digest = decode_source_digest()
    if digest is None or not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[1] == digest:
            return float(parts[2])
    return None


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


# ------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            import tempfile

            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                   "-i", str(self.gpu)]
            import shutil

            if shutil.which("stdbuf"):      # line-buffer so no sample is lost when the sampler stops
                cmd = ["stdbuf", "-oL"] + cmd
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            import signal

            time.sleep(0.25)
            self.proc.send_signal(signal.SIGINT)
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
                self.proc.wait()
            self.out.close()

    def summary(self) -> dict:
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for ln in open(self.path):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) >= 8:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        pw = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "samples": len(rows), "reasons": reasons}


# --------------------------------------------------------------- dist setup
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ the GPU arm
class Step:
    """Device-resident state of one workload and its L-layer decode step.

    A workload with `steps` > 1 (the tiered one) grows every request's context by one
    token per decode step; step t appends position ctx0 + t.  One CUDA graph is captured
    per step index and the timed loop cycles through them.  With scores on, each layer
    also writes its logits and adds its share of the importance score."""

    def __init__(self, w, dev, num_splits: int = 0, early: bool = True, fused_scores: bool = False,
                 host_tier: float = 0.0, host_staged: bool = False, retier: bool = False, planned: bool = True):
        import numpy as np
        import torch

        import paged_gqa_decode_kvd_gb300 as kvd

        self.w, self.dev, self.kvd = w, dev, kvd
        self.early = early   # KVD_EARLY_START: the step's tables and pool are not written by the previous kernel
        self.planned = planned   # one kvd_decode_plan per step, read by every layer's decode (KVD_PLANNED)
        self.L = w.L
        kind = {"bf16": kvd.KVD_BF16, "fp8_e4m3": kvd.KVD_FP8_E4M3, "mixed": kvd.KVD_MIXED, "int4": kvd.KVD_INT4,
                "int2": kvd.KVD_INT2, "angle": kvd.KVD_ANGLE}[w.kv_dtype]
        self.pool = kvd.KVPool(w.L, w.n_kv, w.num_blocks(), kind, device=dev, group_size=w.group_size)
        if w.kv_dtype == "mixed":   # a storage format per physical block
            codes = [kvd.KVD_BF16, kvd.KVD_FP8_E4M3, kvd.KVD_FP8_E5M2]
            fmt = torch.tensor([codes[f] for f in w.block_formats().tolist()], dtype=torch.uint8)
            self.pool.set_block_formats(fmt.to(dev))
        bt = w.block_table()
        self.bt = bt.to(dev)
        self.nsteps = w.steps
        self.lens = [w.seq_lens(t) for t in range(self.nsteps)]
        self.max_len = max(max(x) for x in self.lens)
        ret = w.retain_mask(bt)
        self.retain = None
        if ret is not None:
            self.retain = torch.from_numpy(ret.numpy().astype(np.uint16).view(np.int16)).to(dev)
        # prefill: every position before step 0's append, every layer (setup, untimed)
        first = [c - 1 for c in self.lens[0]]
        for layer in range(w.L):
            for b in range(w.batch):
                if first[b] > 0:
                    k, v = w.kv(layer, b, 0, first[b], dev)
                    kvd.kvd_append_kv(self.pool.handle, layer, k.contiguous(), v.contiguous(),
                                      w.slot_mapping(b, 0, first[b], bt).to(dev))
        self.host_blocks = 0
        self.host_staged = host_staged
        if retier and (host_staged or not w.scores or host_tier <= 0):
            raise ValueError("--retier needs --host-tier, a workload with scores, and in-place T1 reads")
        self.retier_on = retier
        if host_tier > 0:
            bt = self._host_tier(host_tier, bt, retier)
        # per-step inputs: the appended token of every request, q, context lengths
        self.seq, self.slots, self.k_new, self.v_new, self.q = [], [], [], [], []
        for t in range(self.nsteps):
            pos = w.append_pos(t)
            self.seq.append(torch.tensor(self.lens[t], dtype=torch.int32, device=dev))
            self.slots.append(torch.cat([w.slot_mapping(b, pos[b], pos[b] + 1, bt) for b in range(w.batch)]).to(dev))
            kn, vn = [], []
            for layer in range(w.L):
                ks, vs = zip(*[w.kv(layer, b, pos[b], pos[b] + 1, dev) for b in range(w.batch)])
                kn.append(torch.cat(ks))
                vn.append(torch.cat(vs))
            self.k_new.append(torch.stack(kn).contiguous())        # [L][B][n_kv][128]
            self.v_new.append(torch.stack(vn).contiguous())
            self.q.append(torch.stack([w.q(layer, t, dev) for layer in range(w.L)]).contiguous())
        self.out = torch.empty(w.L, w.batch, w.n_q, 128, dtype=torch.bfloat16, device=dev)
        self.splits, nbytes = kvd.kvd_decode_workspace_bytes(self.pool.handle, w.n_q, w.batch, self.max_len,
                                                             num_splits)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.scores = None
        # Score update: by default each layer's share is added on a second stream (the score
        # array is read only when tokens are re-tiered, so no later layer waits for it); the
        # layer's logits and LSE go to a ring of three buffers, and a layer waits only for the
        # score update that last used its slot.  fused_scores: one stream, score update inside
        # the layer's merge launch.
        self.overlap = bool(w.scores) and not fused_scores
        if w.scores:
            nbuf = 3 if self.overlap else 1
            self.lse = torch.empty(nbuf, w.batch, w.n_q, dtype=torch.float32, device=dev)
            self.logits = torch.empty(nbuf, w.batch, w.n_q, self.max_len, dtype=torch.float32, device=dev)
            self.scores = torch.zeros(w.batch, self.max_len, dtype=torch.float32, device=dev)
            if self.overlap:
                self.side = torch.cuda.Stream(device=dev)
                self.score_done = [None] * nbuf
        # per layer: the decode kernel and the merge launch (which also updates the scores when
        # fused), + the score kernel when it runs on its own stream; + the step's plan
        self.launches_per_step = (3 if self.overlap else 2) * w.L + (1 if planned else 0)
        torch.cuda.synchronize()
        err = kvd.kvd_get_device_error(self.pool.handle)
        if err:
            raise RuntimeError(f"device error during setup: {kvd.status_string(err)}")

    def _host_tier(self, frac: float, bt, retier: bool):
        """Host tier (T1): the tier plan, on seeded synthetic scores, picks the frac·nb least
        important unprotected blocks of every request; kvd_tier_reassign gives them host-tier
        ids (free lists, tables and retain mask kept on the host) and kvd_tier_move copies
        them.  In the step the decode kernel reads them in place over the host link, or
        (staged) each layer's host records are copied by a copy-engine DMA on a copy stream,
        two layers ahead of use.  With retier the host tier has room for a reassignment's
        destinations before its sources are freed, and retier() reassigns from the live
        scores."""
        import numpy as np
        import torch

        w, kvd, dev = self.w, self.kvd, self.dev
        g = torch.Generator().manual_seed(w.seed + 7)
        scores = torch.empty(w.batch, self.max_len).exponential_(generator=g).to(dev)
        lens = torch.tensor(self.lens[0], dtype=torch.int32, device=dev)
        mb = bt.shape[1]
        t1 = int(frac * (max(self.lens[0]) + 15) // 16)
        plan = torch.empty(w.batch, mb, dtype=torch.int8, device=dev)
        kvd.kvd_tier_plan(scores, lens, mb, w.protect_prompt, w.protect_recent, t1, plan)
        self.plan_args = (scores, lens, mb, w.protect_prompt, w.protect_recent, t1, plan.clone())
        n_t1 = int((plan == 1).sum())
        if n_t1 == 0:
            return bt
        nb = w.num_blocks()
        nh = 2 * n_t1 if retier else n_t1
        self.pool.attach_host_tier(nh, staged=self.host_staged)
        self.tier_shape = (nb, nh, mb, t1)
        self.bt_host = bt.numpy().astype(np.int32).copy()
        used = np.zeros(nb, bool)
        used[self.bt_host[self.bt_host >= 0]] = True
        free = np.nonzero(~used)[0].astype(np.int32)
        self.hbm_free = np.zeros(nb, np.int32)
        self.hbm_free[:len(free)] = free
        self.hbm_n = len(free)
        self.host_free = np.arange(nb, nb + nh, dtype=np.int32)
        self.host_n = nh
        self.ret_host = None
        if self.retain is not None:
            self.ret_host = np.concatenate([self.retain.cpu().numpy().view(np.uint16), np.full(nh, 0xFFFF, np.uint16)])
        st, frm, to, self.hbm_n, self.host_n = kvd.kvd_tier_reassign(
            nb, nh, plan.cpu().numpy(), self.bt_host, self.hbm_free, self.hbm_n, self.host_free, self.host_n,
            self.ret_host)
        if st != kvd.KVD_OK:
            raise RuntimeError(f"initial tier assignment: {kvd.status_string(st)}")
        self.move_ids = (torch.from_numpy(frm).to(dev), torch.from_numpy(to).to(dev))
        kvd.kvd_tier_move(self.pool.handle, *self.move_ids)
        self.bt = torch.from_numpy(self.bt_host.copy()).to(dev)
        if self.ret_host is not None:
            self.retain = torch.from_numpy(self.ret_host.view(np.int16).copy()).to(dev)
        self.host_blocks = nh
        self.copy = torch.cuda.Stream(device=dev)
        self.host_layer_bytes = nh * w.n_kv * self.pool.record_bytes
        self.plan_dev = torch.empty(w.batch, mb, dtype=torch.int8, device=dev)
        self.retiers, self.retier_moves = 0, 0
        return torch.from_numpy(self.bt_host.copy())

    def t1_bytes_per_step(self) -> int:
        """K/V bytes of the blocks the step reads from the host tier (every layer)."""
        nb = self.tier_shape[0]
        ids = set()
        for b, ln in enumerate(self.lens[0]):
            ids.update(int(x) for x in self.bt_host[b, :(ln + 15) // 16] if x >= nb)
        return len(ids) * self.w.n_kv * self.pool.record_bytes * self.L

    def retier_begin(self, t: int):
        """Start a reassignment (every Δ = 64 steps): the plan from the live importance scores
        and its copy to pinned host memory are queued behind the steps so far; retier_poll
        applies it once the copy has landed, while the GPU keeps running steps."""
        import torch

        w, kvd = self.w, self.kvd
        nb, nh, mb, t1 = self.tier_shape
        if not hasattr(self, "plan_pinned"):
            import numpy as np

            self.plan_pinned = torch.empty(w.batch, mb, dtype=torch.int8, pin_memory=True)
            self.bt_pinned = torch.empty(self.bt_host.shape, dtype=torch.int32, pin_memory=True)
            self.ret_pinned = (None if self.ret_host is None else
                               torch.empty(self.ret_host.shape, dtype=torch.int16, pin_memory=True))
            self.moves_pinned = torch.empty(2, self.bt_host.size, dtype=torch.int32, pin_memory=True)
            self.moves_dev = torch.empty(2, self.bt_host.size, dtype=torch.int32, device=self.dev)
            self.upload_done = None
        self.retier_poll(wait=True)   # one still pending is applied first (the host waits, the GPU has steps queued)
        kvd.kvd_tier_plan(self.scores, self.seq[t], mb, w.protect_prompt, w.protect_recent, t1, self.plan_dev)
        self.plan_pinned.copy_(self.plan_dev, non_blocking=True)
        self.plan_ready = torch.cuda.Event()
        self.plan_ready.record()

    def retier_poll(self, wait: bool = False) -> bool:
        """Apply a started reassignment if its plan has reached the host (or, with wait, once
        it has): host-side reassignment, then the table and retain uploads and the block moves,
        queued in stream order before the next step.  Returns whether one was applied."""
        import numpy as np
        import torch

        if getattr(self, "plan_ready", None) is None or (not wait and not self.plan_ready.query()):
            return False
        self.plan_ready.synchronize()
        self.plan_ready = None
        kvd = self.kvd
        nb, nh, mb, t1 = self.tier_shape
        st, frm, to, self.hbm_n, self.host_n = kvd.kvd_tier_reassign(
            nb, nh, self.plan_pinned.numpy(), self.bt_host, self.hbm_free, self.hbm_n, self.host_free, self.host_n,
            self.ret_host)
        if st != kvd.KVD_OK:
            raise RuntimeError(f"tier reassignment: {kvd.status_string(st)}")
        if len(frm):
            if self.upload_done is not None:
                self.upload_done.synchronize()   # the pinned sources of the last upload are free again
            self.bt_pinned.numpy()[...] = self.bt_host
            self.bt.copy_(self.bt_pinned, non_blocking=True)
            if self.ret_host is not None:
                self.ret_pinned.numpy()[...] = self.ret_host.view(np.int16)
                self.retain.copy_(self.ret_pinned, non_blocking=True)
            n = len(frm)   # pageable sources would synchronise the stream: everything goes through pinned buffers
            self.moves_pinned.numpy()[0, :n] = frm
            self.moves_pinned.numpy()[1, :n] = to
            for r in range(2):   # contiguous rows
                self.moves_dev[r, :n].copy_(self.moves_pinned[r, :n], non_blocking=True)
            kvd.kvd_tier_move(self.pool.handle, self.moves_dev[0, :n], self.moves_dev[1, :n])
            self.upload_done = torch.cuda.Event()
            self.upload_done.record()
        self.retiers += 1
        self.retier_moves += len(frm)
        return True

    def time_host_tier(self, reps: int = 5) -> dict:
        """Host-tier costs measured alone on the copy stream: one step's staging copies, one
        tier plan, and one move of the planned blocks HBM → host (a reassignment that demotes
        them all; the vacated HBM blocks still hold the same records, so repeating it changes
        nothing)."""
        import torch

        kvd, s = self.kvd, self.copy
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def timed(fn, n):
            torch.cuda.synchronize()
            e0.record(s)
            for _ in range(n):
                fn()
            e1.record(s)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / n

        def stage():
            for layer in range(self.L):
                kvd.kvd_tier_prefetch(self.pool.handle, layer, stream=s)

        stage_ms = timed(stage, reps) if self.host_staged else None
        plan_ms = timed(lambda: kvd.kvd_tier_plan(*self.plan_args, stream=s), reps)
        move_ms = timed(lambda: kvd.kvd_tier_move(self.pool.handle, *self.move_ids, stream=s), reps)
        err = kvd.kvd_get_device_error(self.pool.handle)
        if err:
            raise RuntimeError(f"device error in the host-tier timing: {kvd.status_string(err)}")
        step_bytes = self.host_layer_bytes * self.L
        return {"staging_ms_per_step_alone": round(stage_ms, 4) if stage_ms else None,
                "staging_gbs_alone": round(step_bytes / (stage_ms * 1e-3) / 1e9, 1) if stage_ms else None,
                "plan_ms": round(plan_ms, 4), "move_ms": round(move_ms, 4),
                "move_gbs": round(step_bytes / (move_ms * 1e-3) / 1e9, 1),
                "retier_ms_per_step_at_delta_64": round((plan_ms + move_ms) / 64, 4)}

    def _prefetch(self, layer: int):
        import torch

        self.kvd.kvd_tier_prefetch(self.pool.handle, layer, stream=self.copy)
        ev = torch.cuda.Event()
        ev.record(self.copy)
        self.staged[layer] = ev

    def kv_bytes(self, t: int) -> int:
        """Closed-form K/V bytes attended by step t (all layers), FP8 scales excluded."""
        if not hasattr(self, "_kvb"):
            self._kvb = {}
        if t not in self._kvb:
            self._kvb[t] = (self.w.kv_bytes_per_step(t), self.w.scale_bytes_per_step(t))
        return self._kvb[t][0]

    def scale_bytes(self, t: int) -> int:
        self.kv_bytes(t)
        return self._kvb[t][1]

    def layer_call(self, layer: int, t: int = 0, stream=None):
        """One layer's decode: fused append of the new token, attention, split merge, and (with
        scores) this layer's share of the importance score."""
        import torch

        inv = 1.0 / (self.w.L * self.w.n_q)
        if self.overlap:
            i = layer % len(self.score_done)
            cur = stream if stream is not None else torch.cuda.current_stream(self.dev)
            if self.score_done[i] is not None:
                cur.wait_event(self.score_done[i])   # the slot's previous score update is done
            self.kvd.kvd_decode_attn(self.pool.handle, layer, self.q[t][layer], self.bt, self.seq[t], self.max_len,
                                     self.ws, self.out[layer], num_splits=self.splits, retain_mask=self.retain,
                                     lse_out=self.lse[i], logits_out=self.logits[i], k_new=self.k_new[t][layer],
                                     v_new=self.v_new[t][layer], early_start=self.early, planned=self.planned,
                                     stream=cur)
            self.side.wait_stream(cur)
            self.kvd.kvd_accum_scores(self.logits[i], self.lse[i], self.seq[t], inv, self.scores, stream=self.side)
            ev = torch.cuda.Event()
            ev.record(self.side)
            self.score_done[i] = ev
            return
        scores = self.scores is not None
        self.kvd.kvd_decode_attn(self.pool.handle, layer, self.q[t][layer], self.bt, self.seq[t], self.max_len,
                                 self.ws, self.out[layer], num_splits=self.splits, retain_mask=self.retain,
                                 lse_out=self.lse[0] if scores else None, logits_out=self.logits[0] if scores else None,
                                 k_new=self.k_new[t][layer], v_new=self.v_new[t][layer],
                                 scores=self.scores if scores else None, inv_LH=inv,
                                 early_start=self.early, planned=self.planned, stream=stream)

    def decode_kernel_only(self, layer: int, t: int = 0, stream=None):
        """The layer's decode kernel alone (fused append, partials, no merge launch)."""
        scores = self.scores is not None
        self.kvd.kvd_decode_attn(self.pool.handle, layer, self.q[t][layer], self.bt, self.seq[t], self.max_len,
                                 self.ws, None, num_splits=self.splits, retain_mask=self.retain,
                                 logits_out=self.logits[0] if scores else None,
                                 k_new=self.k_new[t][layer], v_new=self.v_new[t][layer], early_start=self.early,
                                 planned=self.planned, stream=stream)

    def plan(self, t: int = 0, stream=None):
        """The step's plan (block tables, lengths and retain mask are the same for all its layers)."""
        if self.planned:
            self.kvd.kvd_decode_plan(self.pool.handle, self.w.n_q, self.bt, self.seq[t], self.max_len, self.ws,
                                     num_splits=self.splits, retain_mask=self.retain, stream=stream)

    def capture_decode_only(self):
        import torch

        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.plan(0)
            for layer in range(self.L):
                self.decode_kernel_only(layer)
        torch.cuda.synchronize()
        return g

    def run(self, t: int = 0, stream=None):
        import torch

        cur = stream if stream is not None else torch.cuda.current_stream(self.dev)
        if self.overlap:
            self.score_done = [None] * len(self.score_done)   # a step depends on nothing of the last
        staged = self.host_blocks and self.host_staged
        self.plan(t, cur)
        if staged:   # staging slots 0 and 1 are free at the start of a step
            self.copy.wait_stream(cur)
            self.staged = [None] * self.L
            for layer in range(min(2, self.L)):
                self._prefetch(layer)
        for layer in range(self.L):
            if staged:
                cur.wait_event(self.staged[layer])
            self.layer_call(layer, t, stream)
            if staged and layer + 2 < self.L:   # refill this layer's slot once it is read
                done = torch.cuda.Event()
                done.record(cur)
                self.copy.wait_event(done)
                self._prefetch(layer + 2)
        if self.overlap:   # the step ends when its last score update has
            cur.wait_stream(self.side)

    def capture(self):
        import torch

        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(s):
            self.run(0)
        torch.cuda.current_stream(self.dev).wait_stream(s)
        torch.cuda.synchronize()
        graphs = []
        for t in range(self.nsteps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.run(t)
            graphs.append(g)
        torch.cuda.synchronize()
        return graphs




# ------------------------------------------------------------------ shared descriptions
def workload_config(w) -> dict:
    """The `config` of a JSON line: the workload and its sizes, identical for both arms."""
    return {"workload": f"{w.name}: {w.description}", "layers": w.L, "batch": w.batch, "n_q": w.n_q,
            "n_kv": w.n_kv, "d_h": w.d_h, "kv_dtype": w.kv_dtype,
            "context": w.seq_lens(0)[:4] if w.batch > 4 else w.seq_lens(0),
            "kv_bytes_per_step": w.kv_bytes_per_step(), "scale_bytes_per_step": w.scale_bytes_per_step(),
            "group_size": w.group_size or None,
            "decode_steps_cycled": w.steps, "scores": bool(w.scores), "seed": w.seed,
            "l2": "inputs larger than L2 (KV pool streamed every step)"}


def read_stream_peak(dev, gib: int = 4, reps: int = 10) -> dict:
    """Read-only HBM bandwidth: kvd_measure_read_stream over a `gib` GiB buffer, best of `reps`
    CUDA-event-timed passes after 3 warm-up passes (the buffer is 30x the L2)."""
    import torch

    import paged_gqa_decode_kvd_gb300 as kvd

    buf = torch.empty(gib << 30, dtype=torch.uint8, device=dev)
    buf.fill_(0x5A)
    sink = torch.empty(1 << 15, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev)
    for _ in range(3):
        kvd.kvd_measure_read_stream(buf, sink, stream=s)
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        kvd.kvd_measure_read_stream(buf, sink, stream=s)
        e1.record(s)
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    nbytes = buf.numel()
    del buf, sink
    torch.cuda.empty_cache()
    return {"gbs": round(nbytes / (best * 1e-3) / 1e9, 1), "bytes": nbytes, "best_ms": round(best, 4),
            "how": f"kvd_measure_read_stream: {gib} GiB read once with 16-byte streaming loads, best of {reps}"}


# ------------------------------------------------------------------ the GPU arm
def gpu_workload(args, w, rank, world, local, peaks, headline: bool) -> dict:
    """Time one workload's decode steps (CUDA graph per step, W warm-up + K timed replays,
    events on the stream, clocks sampled), its decode kernel alone (roofline) and, for the
    headline line, the end-to-end steps through the public API with host copies."""
    import torch

    dev = torch.device("cuda", local)
    st = Step(w, dev, args.num_splits, early=not args.no_early_start, fused_scores=args.fused_scores,
              host_tier=args.host_tier if headline else 0.0, host_staged=args.host_tier_staged,
              retier=args.retier and headline, planned=not args.no_plan)
    graphs = st.capture()
    stream = torch.cuda.current_stream(dev)
    steps = args.steps
    kv_bytes = sum(st.kv_bytes(t % st.nsteps) for t in range(steps)) / steps

    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        for i in range(args.warmup):
            if st.retier_on:
                st.retier_poll()
                if i % st.nsteps == 0 and i > 0:
                    st.retier_begin(0)
            graphs[i % st.nsteps].replay()
        if st.retier_on:
            st.retier_poll(wait=True)
        torch.cuda.synchronize()
        if st.retier_on:
            st.retiers, st.retier_moves = 0, 0
        barrier(world)
        t0.record(stream)
        for i in range(steps):
            if st.retier_on:   # every Δ = 64 steps (the step cycle), applied without stopping the GPU
                st.retier_poll()
                if i % st.nsteps == 0 and i > 0:
                    st.retier_begin(0)
            graphs[i % st.nsteps].replay()
        if st.retier_on:
            st.retier_poll(wait=True)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = t0.elapsed_time(t1)
    ms_max = max_over_ranks(ms, world)
    ms_per_step = ms_max / steps
    value = kv_bytes * world / (ms_per_step * 1e-3) / 1e9
    err = st.kvd.kvd_get_device_error(st.pool.handle)
    if err:
        raise RuntimeError(f"device error after timed steps of {w.name}: {st.kvd.status_string(err)}")

    # per-launch time of the dominant kernel (the decode kernel), from a graph of its L
    # launches alone replayed on the same stream, so host enqueue time cannot inflate it
    dgraph = st.capture_decode_only()
    dgraph.replay()
    torch.cuda.synchronize()
    reps = max(3, min(50, steps // 4))
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for _ in range(reps):
        dgraph.replay()
    d1.record(stream)
    torch.cuda.synchronize()
    dec_ms = d0.elapsed_time(d1) / (reps * st.L)
    layer_bytes = (st.kv_bytes(0) + st.scale_bytes(0)) / w.L
    achieved = layer_bytes / (dec_ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": (args.traffic if args.traffic is not None else
                        recorded_traffic(w.name) if not args.layers and not args.context else None),
            "kernel": "kvd::decode_kernel", "peak_source": peaks["source"] + " (copy, MEASURED_PEAKS.json hbm_gbs)",
            "bytes_per_launch": layer_bytes, "launch_ms": round(dec_ms, 5)}
    if peaks.get("read_gbs"):
        roof["frac_of_read_peak"] = round(achieved / peaks["read_gbs"], 4)
    del dgraph

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"bf16": "bf16", "fp8_e4m3": "fp8_e4m3",
                                       "mixed": "mixed: bf16 / fp8_e4m3 / fp8_e5m2 per block",
                                       "int4": f"int4 (group {w.group_size}, f16 scale and zero)",
                                       "int2": f"int2 (group {w.group_size}, f16 scale and zero)",
                                       "angle": "angle-domain keys (fp8_e4m3 direction codes), fp8_e4m3 values"}[
                                           w.kv_dtype],
        "data": "synthetic (seeded counter-hash generator)",
        "config": workload_config(w),
        "launch": {"num_splits": st.splits, "early_start": st.early, "step_plan": st.planned,
                   # the decode kernel balances the last sixth of every split's range at run time for
                   # planned BF16 calls whose ranges hold at least 192 blocks (computed here the same way)
                   "run_time_balancing": bool(st.planned and w.kv_dtype == "bf16" and
                                              -(-sum(-(-n // w.block_size) for n in w.seq_lens(0)) * w.n_kv
                                                // st.splits) >= 192),
                   "score_update": ("second stream (off the layer chain)" if st.overlap else
                                    "fused into the call's epilogue launch" if w.scores else None),
                   "parallelism": f"replicas x{world}"},
        "steps_per_s": round(1e3 / ms_per_step, 2),
        "hbm_frac_of_measured": round(value / world / peaks["hbm_gbs"], 4),
        "hbm_frac_of_datasheet_8tbs": round(value / world / 8000.0, 4),
        "roofline": roof,
        "gpu_launches": st.launches_per_step * steps,
        "clocks": clk.summary(),
    }
    if peaks.get("read_gbs"):
        line["hbm_frac_of_read_peak"] = round(value / world / peaks["read_gbs"], 4)
    if st.host_blocks:
        line["launch"]["host_tier"] = {
            "fraction": args.host_tier, "host_blocks": st.host_blocks,
            "host_bytes_per_step": st.t1_bytes_per_step(),
            "retier": None if not st.retier_on else {
                "every_steps": st.nsteps, "in_timed_region": st.retiers, "blocks_moved": st.retier_moves},
            "read": ("staged: copy-engine DMA per layer on a copy stream, two layers ahead"
                     if st.host_staged else "direct: the decode kernel reads host records in place"),
            **st.time_host_tier()}
    if headline:
        line["e2e"] = e2e_steps(st, args, world)
    del graphs
    st.pool.close()
    return line


def e2e_steps(st, args, world) -> dict:
    """The same steps end to end through the public API: per step, the step's q and new K/V
    copied from pinned host memory, one kvd_decode_attn call per layer issued from the host
    (no graph), and the outputs copied back to pinned host memory; K steps after W warm-up."""
    import torch

    stream = torch.cuda.current_stream(st.dev)
    h_q = [q.cpu().pin_memory() for q in st.q]
    h_k = [k.cpu().pin_memory() for k in st.k_new]
    h_v = [v.cpu().pin_memory() for v in st.v_new]
    h_out = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()

    def one(t):
        i = t % st.nsteps
        st.q[i].copy_(h_q[i], non_blocking=True)
        st.k_new[i].copy_(h_k[i], non_blocking=True)
        st.v_new[i].copy_(h_v[i], non_blocking=True)
        st.run(i)
        h_out.copy_(st.out, non_blocking=True)

    for t in range(args.warmup):
        one(t)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for t in range(args.steps):
        one(t)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    i = 0
    h2d = (h_q[i].numel() * h_q[i].element_size() + h_k[i].numel() * h_k[i].element_size()
           + h_v[i].numel() * h_v[i].element_size())
    d2h = h_out.numel() * h_out.element_size()
    kv = sum(st.kv_bytes(t % st.nsteps) for t in range(args.steps)) / args.steps
    return {"value": round(kv * world / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
            "how": "eager per-layer kvd_decode_attn calls from the host (no graph), the step's inputs "
                   "copied from pinned host memory and its outputs back, every step"}


EXTRA_WORKLOADS = ("ragged", "llama70b_fp8", "tiered", "llama8b_mixed", "llama70b_int4", "llama70b_int2",
                   "llama70b_angle")


def gpu_arm(args, w, rank, world, local):
    import gc

    import torch

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = measured_peaks()
    if not args.no_read_peak:
        peaks["read"] = read_stream_peak(dev)
        peaks["read_gbs"] = peaks["read"]["gbs"]
    line = gpu_workload(args, w, rank, world, local, peaks, headline=True)
    if "read" in peaks:
        line["hbm_read_peak"] = peaks["read"]
    # the default run also measures the other full-size workloads on one GPU (the headline
    # `value` stays the default workload's)
    if world == 1 and args.workload == "llama8b" and not args.only:
        others = {}
        for name in EXTRA_WORKLOADS:
            gc.collect()
            torch.cuda.empty_cache()
            from kvd_inputs import get

            sub = gpu_workload(args, get(name, args.seed), rank, world, local, peaks, headline=False)
            for k in ("metric", "unit", "n_gpus", "warmup", "higher_is_better", "scaling", "vs_baseline", "data"):
                sub.pop(k, None)
            others[name] = sub
        line["workloads"] = others
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    return line


# ------------------------------------------------------------------ the CPU oracle arm
def _oracle_unit(w, layer: int, b: int, kf, vf, q, fmt=None):
    """The oracle on one (layer, request) unit: append of its context into the oracle's own pool,
    then decode of all its query heads (fp64).  fmt: a mixed pool's formats of the request's
    blocks, in table order."""
    import numpy as np

    import oracle

    n = kf.shape[0]
    nblk = -(-n // 16)
    slots = np.arange(n, dtype=np.int64)
    table = np.arange(nblk, dtype=np.int32)[None, :]
    if fmt is not None:
        pool = oracle.OraclePool(nblk, w.n_kv, w.d_h, 16, block_fmt=fmt)
    elif w.lowbit:
        pool = oracle.OraclePool(nblk, w.n_kv, w.d_h, 16, lowbit=w.lowbit)
    elif w.kv_dtype == "angle":
        pool = oracle.OraclePool(nblk, w.n_kv, w.d_h, 16, angle=True)
        q = oracle.angle_query(q)
    else:
        pool = oracle.OraclePool(nblk, w.n_kv, w.d_h, 16, w.kv_dtype != "bf16")
    pool.append(kf, vf, slots)
    oracle.decode(pool, q, w.n_q, table, [n])


def _unit_inputs(w, b: int):
    """Inputs of the (layer 0, request b) unit: K, V, q, the block formats (mixed pools) and the
    unit's closed-form K/V bytes."""
    n = w.seq_lens(0)[b]
    k, v = w.kv(0, b, 0, n)
    fmt = None
    if w.kv_dtype == "mixed":
        nblk = -(-n // 16)
        fmt = w.block_formats()[w.block_table()[b, :nblk].numpy()]
        wide = int((fmt == 0).sum()) * 16 - (16 * nblk - n if fmt[-1] == 0 else 0)
        nbytes = 2 * w.n_kv * w.d_h * (2 * wide + (n - wide))
    else:
        nbytes = kv_bytes_per_token(1, w.n_kv, w.d_h, w.w_kv) * n
    return k.float().numpy(), v.float().numpy(), w.q(0, 0)[b:b + 1].float().numpy(), fmt, nbytes


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(w, threads: int, budget_s: float) -> dict:
    """Time the oracle (as it stands) on `threads` host threads, each running whole (layer 0,
    request b) units of the workload (b = thread index mod batch), until `budget_s` seconds of
    wall time have passed; returns KV bytes attended per second over the units completed."""
    import concurrent.futures as cf

    import oracle

    oracle.build()
    ins = [_unit_inputs(w, b % w.batch) for b in range(min(threads, w.batch))]
    per_unit = [x[4] for x in ins]

    def worker(i):
        units, done = 0, 0.0
        t0 = time.perf_counter()
        while True:
            _oracle_unit(w, 0, i, *ins[i % len(ins)][:4])
            units += 1
            done += per_unit[i % len(ins)]
            if time.perf_counter() - t0 >= budget_s:
                return units, done

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:   # ctypes releases the GIL in the C oracle
        res = list(ex.map(worker, range(threads)))
    wall = time.perf_counter() - t0
    units = sum(r[0] for r in res)
    nbytes = sum(r[1] for r in res)
    return {"gbs": nbytes / wall / 1e9, "units": units, "wall_s": wall, "bytes": nbytes}


def cpu_baseline(w, budget_s: float = 15.0) -> dict:
    """The fp64 oracle timed on the host cores on a bounded sample of the workload: whole
    (layer 0, request) units, first on one thread, then on every core the process may use."""
    n = host_threads()
    one = oracle_sample(w, 1, budget_s / 2)
    allc = oracle_sample(w, n, budget_s / 2)
    return {"value": round(allc["gbs"], 4), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{allc['units']} whole (layer 0, request) units of {w.name} (append + decode of every "
                      f"query head, fp64) on {n} host threads in {allc['wall_s']:.1f} s; KV bytes attended / wall time",
            "steps_per_s": round(allc["gbs"] * 1e9 / w.kv_bytes_per_step(), 6),
            "single_thread": {"value": round(one["gbs"], 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{one['units']} units on one thread in {one['wall_s']:.1f} s"}}


def reference_arm(args, w, rank, world):
    """The oracle as the reference arm: each step is one bounded sample of the workload, one
    whole (layer 0, request b) unit per host thread, run in parallel; value = KV bytes the
    sample attended / its wall time (the rate is measured, not extrapolated)."""
    if rank != 0:
        return None
    import oracle

    oracle.build()
    n = host_threads()
    ins = [_unit_inputs(w, b % w.batch) for b in range(min(n, w.batch))]
    import concurrent.futures as cf

    def sample():
        t0 = time.perf_counter()
        with cf.ThreadPoolExecutor(max_workers=n) as ex:
            list(ex.map(lambda i: _oracle_unit(w, 0, i, *ins[i % len(ins)][:4]), range(n)))
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        sample()
    walls = [sample() for _ in range(args.steps)]
    per_sample = sum(ins[i % len(ins)][4] for i in range(n))
    total_s = sum(walls)
    gbs = per_sample * args.steps / total_s / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total_s / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded counter-hash generator)", "config": workload_config(w),
            "step": f"one bounded sample: {n} whole (layer 0, request) units of {w.name} in parallel on {n} host "
                    f"threads ({per_sample / 1e6:.1f} MB of KV attended)",
            "extrapolated": False,
            "full_step_s_at_this_rate": round(w.kv_bytes_per_step() / (gbs * 1e9), 1),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
                             "sample": f"{args.steps} samples of {n} (layer 0, request) units, fp64"},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--only", action="store_true",
                    help="time the chosen workload alone (the default run also times the ragged, 70B FP8, "
                         "tiered, mixed-precision, 70B low-bit and 70B angle-domain workloads)")
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (small profiling captures)")
    ap.add_argument("--context", type=int, default=0, help="override every request's context (size sweeps)")
    ap.add_argument("--group-size", type=int, default=0,
                    help="low-bit workloads: values per scale group (32, 64 or 128) instead of the workload's")
    ap.add_argument("--no-early-start", action="store_true", help="launch the decode kernel without KVD_EARLY_START")
    ap.add_argument("--no-plan", action="store_true",
                    help="no step plan: every layer's decode kernel derives its split from the lengths and tables")
    ap.add_argument("--fused-scores", action="store_true",
                    help="score update inside each layer's epilogue launch (one stream) instead of on a second stream")
    ap.add_argument("--host-tier", type=float, default=0.0,
                    help="fraction of each request's blocks the tier plan moves to the host tier (T1)")
    ap.add_argument("--retier", action="store_true",
                    help="reassign tiers from the live scores every 64 steps inside the timed loop")
    ap.add_argument("--host-tier-staged", action="store_true",
                    help="stage each layer's host-tier records in HBM (DMA) instead of reading them in place")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=16.0, help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-read-peak", action="store_true", help="skip the read-only HBM stream measurement")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes read+write per decode launch from an ncu capture of the current kernel")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    from kvd_inputs import get

    rank, world, local = dist_env()
    w = get(args.workload, args.seed)
    if args.layers:
        w.L = args.layers
        w.description += f" [reduced to {args.layers} layers for profiling]"
        args.only = True
    if args.context:
        if w.steps > 1:
            ap.error("--context applies to fixed-context workloads only")
        w._ctx0 = [args.context] * w.batch
        w.description += f" [context set to {args.context} for a size sweep]"
        args.only = True
    if args.group_size:
        if not w.lowbit:
            ap.error("--group-size applies to the low-bit workloads only")
        w.group_size = args.group_size
        w.description += f" [group size set to {args.group_size}]"
        args.only = True
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if args.impl == "gb300" else "gloo")
    if args.impl == "reference":
        line = reference_arm(args, w, rank, world)
    else:
        line = gpu_arm(args, w, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
