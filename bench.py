"""Benchmark of the paged KV-cache hot path on GB300.

One step = one pass of the path over one batch: build the slot mapping of
the step's new tokens, append them to the paged cache (kv_append), then run
paged_decode over every sequence.  The default workload is the
long-context fp8 decode step (batch 16, 64 q / 8 kv heads, head_dim 128,
block 32, contexts U{16384..32768}, e4m3 cache with per-kv-head scales, bf16
q); the GQA bf16, 3-bit MHA, mixed prefill+decode append and the other
workloads are measured in the same run and reported under "workloads", each
with its own roofline block.

Every decode workload's timed step is checked: after the timed replays the
step graph runs once more, its output and the cache it leaves are copied to
the host, and the oracle (the CPU-baseline leg) re-applies the step's append
to a copy of that cache (bit-exact: nothing may change) and decodes every
(sequence, head) over it; the largest absolute error against the stated
tolerance is reported under "parity".

value = algorithmic bytes of the step / device time of the step (GB/s), with
the inputs resident in HBM and L2 flushed between steps (a 256 MiB write
outside the timed events).  e2e = the same metric through the public API
with the step's inputs in pinned host memory, copied in and the output
copied out inside the timed region.  The CPU oracle is timed on a bounded
sample of the same workload (cpu_baseline); ``--impl reference`` times the
oracle alone as the reference arm.

Multi-GPU (torchrun): every rank runs an independent replica of the
workload (the path has no exchange step); value = total bytes of all ranks /
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
# sources of the persistent decode kernel (the automatic plan's); a recorded
# ncu traffic figure is only used while these are unchanged
DECODE_SOURCES = ("paged_kv_cache_num_gb300/csrc/decode_tma.cu",
                  "paged_kv_cache_num_gb300/csrc/decode_tma_kernel.cuh",
                  "paged_kv_cache_num_gb300/csrc/decode_tma_xv.cu",
                  "paged_kv_cache_num_gb300/csrc/pkv_ptx.cuh",
                  "paged_kv_cache_num_gb300/csrc/pkv_device.cuh")


class L2Flush:
    """Between timed steps: write a 256 MiB buffer (evicts L2), then read a
    512 MiB buffer so the dirty lines of that write are written back before
    the next timed region starts instead of inside it."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(2 * L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def zero_(self):
        self.w.zero_()
        self.r.sum()
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def job_throughput(pg, bytes_local, ms_local, device):
    """Whole-job throughput over all ranks: the bytes every rank processed
    divided by the slowest rank's time (max over ranks).  Returns
    (ms_max, GB/s).  ``pg`` is torch.distributed (any backend) or None."""
    ms_t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    b_t = torch.tensor([float(bytes_local)], dtype=torch.float64, device=device)
    if pg is not None:
        pg.all_reduce(ms_t, op=pg.ReduceOp.MAX)
        pg.all_reduce(b_t, op=pg.ReduceOp.SUM)
    ms_max = float(ms_t.item())
    return ms_max, float(b_t.item()) / (ms_max * 1e-3) / 1e9


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(*files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic(kernel_tag, src_hash):
    """dram bytes per launch recorded by an ncu capture (profiles/), if the
    kernel source has not changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = dict(kv.split("=", 1) for kv in line.strip().split() if "=" in kv)
        if parts.get("kernel") == kernel_tag and parts.get("src") == src_hash:
            try:
                return float(parts["dram_bytes_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *a):
        time.sleep(0.15)
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
                self.lines = [l for l in out.splitlines() if l.strip()]
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- workloads

def algorithmic_bytes(w, decode=True, append=True):
    """Bytes the method must move (not the dense pool):
    decode: sum_b ctx_b * Hkv * (K row + V row + 3-bit metadata) + q + out +
            block-table entries read + context_lens;
    append: per real new token Hkv * (2 source rows + 2 cache rows + metadata)
            + its slot (8 B) and (request, position) (8 B)."""
    D, Hkv, BS = w.head_dim, w.num_kv_heads, w.block_size
    row = {"f16": 2 * D, "bf16": 2 * D, "e4m3": D, "e5m2": D, "i8": D, "u3": 3 * D // 8}[w.cache_kind]
    # per cached row and K/V: 3-bit scale + zero, or a per-token fp32 scale
    meta = 3 if w.cache_kind == "u3" else (4 if w.scale_mode == "token" else 0)
    total = 0
    if decode and w.q is not None:
        ctx = w.context_lens.to(torch.int64).cpu()
        nblk = int(((ctx + BS - 1) // BS).sum())
        total += int(ctx.sum()) * Hkv * 2 * (row + meta)
        total += 2 * w.q.numel() * 2                       # q in, out
        total += nblk * 4 + w.batch * 4
        if w.scale_mode == "block":                        # each block's K and V scales
            total += nblk * Hkv * 2 * 4
    if append:
        n_real = int((w.new_pos >= 0).sum())
        # a per-token scale is read with the row and written at its slot
        meta_app = meta + (4 if w.scale_mode == "token" else 0)
        total += n_real * Hkv * 2 * (2 * D + row + meta_app) + n_real * 16
    return total


def fill_row_bytes(w):
    """Algorithmic bytes of one token of a context-fill append (slots given):
    its K and V source rows read, its cache rows (and 3-bit scale / zero)
    written, its slot read."""
    D, Hkv = w.head_dim, w.num_kv_heads
    row = {"f16": 2 * D, "bf16": 2 * D, "e4m3": D, "e5m2": D, "i8": D, "u3": 3 * D // 8}[w.cache_kind]
    meta = 3 if w.cache_kind == "u3" else 0
    return Hkv * 2 * (2 * D + row + meta) + 8


def make_workload(name, device, rank=0):
    """The named workload; rank r > 0 (a replica under torchrun) draws an
    independent instance of the same recipe (seed + 1000 r)."""
    seed = W.SEEDS[name] + 1000 * rank
    if name == "gqa_bf16":
        return W.gqa_bf16(device=device, seed=seed)
    if name == "fp8_long":
        return W.fp8_long(device=device, seed=seed)
    if name == "fp8_long_e5m2":
        return W.fp8_long(device=device, seed=seed, fp8="e5m2")
    if name == "i8_long":
        return W.fp8_long(device=device, seed=seed, fp8="i8")
    if name == "fp8_long_token_scales":
        return W.fp8_long(device=device, seed=seed, scales="token")
    if name == "fp8_long_block_scales":
        return W.fp8_long(device=device, seed=seed, scales="block")
    if name == "gqa_bf16_xvec":
        return W.gqa_bf16(device=device, seed=seed, layout="xvec")
    if name == "fp8_long_xvec":
        return W.fp8_long(device=device, seed=seed, layout="xvec")
    if name == "fp8_long_g16":
        return W.fp8_long(device=device, seed=seed, num_heads=128)
    if name == "gqa_bf16_g16":
        return W.gqa_bf16(device=device, seed=seed, num_heads=128)
    if name == "fp8_long_d64":
        return W.fp8_long(device=device, seed=seed, head_dim=64)
    if name == "u3_mha":
        return W.u3_mha(device=device, seed=seed)
    if name in ("u3_g16", "u3_g8"):
        return W.u3_mha(device=device, seed=seed, batch=16, ctx_lo=8192, ctx_hi=32768,
                        num_heads=128 if name == "u3_g16" else 64, num_kv_heads=8)
    if name == "mixed_append":
        return W.mixed_append(device=device, seed=seed)
    if name == "mha_short":
        return W.mha_short(device=device, seed=seed)
    if name == "tiny_fp16":
        return W.tiny(device=device)
    raise ValueError(name)


class Step:
    """Device-resident state of one workload and its step."""

    def __init__(self, w, pkv, num_splits=0):
        self.w, self.pkv, self.num_splits = w, pkv, num_splits
        dev = w.new_req.device
        self.cache = pkv.KVCache.allocate(
            w.cache_kind, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, device=dev,
            k_scale=w.k_scale, v_scale=w.v_scale, fill=0, scale_mode=w.scale_mode,
            k_scales=w.k_block_scale, v_scales=w.v_block_scale, layout=w.layout)
        self.tok = w.scale_mode == "token"
        if w.k_cache0 is not None:
            self.cache.k_cache.copy_(W.storage(w.k_cache0, w.layout))
            self.cache.v_cache.copy_(W.storage(w.v_cache0, w.layout))
            w.k_cache0 = w.v_cache0 = None      # release the staging copies
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.fill = None
        if w.fill_req is not None:            # context fill (setup, not timed)
            ch = 1 << 18
            first = None
            for i in range(0, w.fill_req.shape[0], ch):
                sm = pkv.slot_mapping(w.block_tables, w.fill_req[i:i + ch], w.fill_pos[i:i + ch],
                                      w.block_size, err_flag=self.err)
                if self.tok:
                    pkv.kv_append_scaled(w.k_fill[i:i + ch], w.v_fill[i:i + ch],
                                         w.k_fill_scale[i:i + ch], w.v_fill_scale[i:i + ch], sm,
                                         self.cache, err_flag=self.err)
                elif first is None:
                    first = (w.k_fill[i:i + ch], w.v_fill[i:i + ch], sm)
                    pkv.kv_append(*first, self.cache, err_flag=self.err)
                else:
                    pkv.kv_append(w.k_fill[i:i + ch], w.v_fill[i:i + ch], sm, self.cache,
                                  err_flag=self.err)
            if first is not None:
                # the first chunk's append again (it writes the same bytes),
                # timed alone: a prefill-sized quantising append
                ts = []
                for _ in range(3):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    pkv.kv_append(*first, self.cache, err_flag=self.err)
                    e1.record()
                    torch.cuda.synchronize()
                    ts.append(e0.elapsed_time(e1))
                n = int(first[2].shape[0])
                self.fill = {"tokens": n, "ms": min(ts),
                             "bytes": n * fill_row_bytes(w)}
                del first
            w.k_fill = w.v_fill = w.fill_req = w.fill_pos = None
            w.k_fill_scale = w.v_fill_scale = None
        self.slots = torch.empty(w.new_req.shape[0], dtype=torch.int64, device=dev)
        self.out = torch.empty_like(w.q) if w.q is not None else None
        self.ws = None
        self.fused = w.q is not None and not self.tok
        self.launches = 1 if self.fused else 2     # (slot computation +) append
        if w.q is not None:
            n = pkv.decode_workspace_bytes(w.q, self.cache, w.block_tables, num_splits)
            self.ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
            self.launches += pkv.decode_launches(w.q, self.cache, w.block_tables, num_splits)
        torch.cuda.synchronize()

    def append(self, req=None, pos=None, k=None, v=None):
        w, pkv = self.w, self.pkv
        pkv.slot_mapping(w.block_tables, w.new_req if req is None else req,
                         w.new_pos if pos is None else pos, w.block_size, out=self.slots,
                         err_flag=self.err)
        if self.tok:
            pkv.kv_append_scaled(w.k_new if k is None else k, w.v_new if v is None else v,
                                 w.k_new_scale, w.v_new_scale, self.slots, self.cache,
                                 err_flag=self.err)
        else:
            pkv.kv_append(w.k_new if k is None else k, w.v_new if v is None else v, self.slots,
                          self.cache, err_flag=self.err)

    def decode(self, q=None):
        w = self.w
        if w.q is None:
            return
        self.pkv.paged_decode(w.q if q is None else q, self.cache, w.block_tables,
                              w.context_lens, sm_scale=w.sm_scale, out=self.out,
                              num_splits=self.num_splits, workspace=self.ws, err_flag=self.err)

    def run(self):
        """One whole step through the public API: pkv_decode_step (slot
        computation fused into the append kernel, then decode) where it
        applies, else the separate calls (append-only workloads, per-token
        scales, which need pkv_kv_append_scaled)."""
        w = self.w
        if self.fused:
            self.pkv.decode_step(w.k_new, w.v_new, w.new_req, w.new_pos, w.q, self.cache,
                                 w.block_tables, w.context_lens, sm_scale=w.sm_scale, out=self.out,
                                 slots=self.slots, num_splits=self.num_splits, workspace=self.ws,
                                 err_flag=self.err)
        else:
            self.append()
            self.decode()

    def capture(self):
        """Record the step's launches (see run) as one CUDA graph, and its
        append (slot_mapping + kv_append) and decode parts as two more;
        replays run the same kernels on the same buffers without the Python /
        ctypes launch overhead."""
        self.run()                             # warm: function attributes, maps
        torch.cuda.synchronize()
        self.g_step = torch.cuda.CUDAGraph()
        self.g_app, self.g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_step):
            self.run()
        with torch.cuda.graph(self.g_app):
            self.append()
        if self.w.q is not None:          # append-only workloads have no decode part
            with torch.cuda.graph(self.g_dec):
                self.decode()
        torch.cuda.synchronize()

    def replay_step(self):
        self.g_step.replay()

    def replay_append(self):
        self.g_app.replay()

    def replay_decode(self):
        if self.w.q is not None:
            self.g_dec.replay()


def time_pack3_bijection(pkv, dev, flush, reps=20):
    """Every 24-bit octet state (2^24 octets, 134 MB of codes) packed and
    unpacked on the GPU: per-call device times, and whether the round trip
    and the closed form pack(v) = the 3 little-endian bytes of the state
    index held for every state."""
    vals = W.all_octets(dev).reshape(-1)
    n = vals.numel() // 8
    packed = torch.empty(n * 3, dtype=torch.uint8, device=dev)
    back = torch.empty_like(vals)
    words = torch.empty(n // 4 * 3, dtype=torch.int32, device=dev)
    back_w = torch.empty_like(vals)
    for _ in range(3):
        pkv.pack3(vals, packed)
        pkv.unpack3(packed, back)
    torch.cuda.synchronize()
    ok = bool(torch.equal(back, vals))
    idx = torch.arange(n, dtype=torch.int64, device=dev)
    closed = torch.stack([idx & 0xFF, (idx >> 8) & 0xFF, idx >> 16], 1).to(torch.uint8).reshape(-1)
    ok = ok and bool(torch.equal(packed, closed))
    words.view(torch.uint8).copy_(packed)
    pkv.unpack3_words(words, back_w)
    torch.cuda.synchronize()
    ok = ok and bool(torch.equal(back_w, vals))
    del idx, closed
    t = {"pack": [], "unpack": [], "unpack_words": []}
    for _ in range(reps):
        for name, fn in (("pack", lambda: pkv.pack3(vals, packed)),
                         ("unpack", lambda: pkv.unpack3(packed, back)),
                         ("unpack_words", lambda: pkv.unpack3_words(words, back_w))):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            t[name].append(e0.elapsed_time(e1))
    nbytes = vals.numel() + packed.numel()
    res = {"octets": n, "bijection_and_closed_form_ok": ok}
    for name, v in t.items():
        ms = float(np.median(v))
        res[name + "_ms"] = round(ms, 4)
        res[name + "_gbs"] = round(nbytes / (ms * 1e-3) / 1e9, 1)
    res["pages_context"] = "2^24 check: 0.91 s on a CPU, 1982.2 ms in Triton on an RTX 3060 Laptop GPU"
    return res


def time_graph(replay, steps, flush):
    """CUDA-event times (ms) of `steps` replays, L2 flushed before each."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        flush.zero_()
        a.record()
        replay()
        b.record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def time_steps(step, steps, warmup, flush, parts=True):
    """Per-step CUDA-event times (ms) of `steps` replays of the one-graph
    step after `warmup`, L2 flushed before each; with `parts`, then as many
    replays of its append and decode parts alone: (step, append, decode)."""
    if not hasattr(step, "g_step"):
        step.capture()
    for _ in range(warmup):
        flush.zero_()
        step.replay_step()
    torch.cuda.synchronize()
    tot = time_graph(step.replay_step, steps, flush)
    if not parts:
        return tot, None, None
    app = time_graph(step.replay_append, steps, flush)
    dec = time_graph(step.replay_decode, steps, flush) if step.w.q is not None else [0.0]
    return tot, app, dec


# ---------------------------------------------------------------- configs

def workload_config(w, name, ws):
    """The workload a bench line measures (both arms print this)."""
    return {"workload": name, "batch": w.batch, "num_heads": w.num_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "context": w.extra.get("context"),
            "cache_dtype": w.cache_kind, "q_dtype": str(w.dtype).replace("torch.", ""),
            "scale_mode": w.scale_mode, "layout": w.layout,
            "new_tokens": int((w.new_pos >= 0).sum()),
            "parallelism": "replicas" if ws > 1 else "single"}


def decode_roofline(name, dec_bytes, dec_ms, peak, peak_src, num_splits=0):
    gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    # recorded traffic is the persistent kernel's (the automatic plan)
    traffic = (profile_traffic("paged_decode:" + name, source_hash(*DECODE_SOURCES))
               if num_splits == 0 else None)
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
            "frac": round(gbs / peak, 4), "traffic": traffic,
            "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)" if peak_src ==
            "measured" else "fallback 6.8 TB/s",
            "kernel": "paged_decode (decode kernel + split-K merge, one C-ABI call)",
            "algorithmic_bytes_per_launch": dec_bytes}


# ---------------------------------------------------------------- timed-output check

def cache_host_logical(cache, layout):
    """Host copies of the cache arrays in the logical [P, BS, Hkv, ...] order
    (x-vectorised storage rearranged back), as numpy bit patterns."""
    d = {}
    for name in ("k_cache", "v_cache", "k_qscale", "k_qzero", "v_qscale", "v_qzero", "k_scales",
                 "v_scales"):
        t = getattr(cache, name)
        if t is None:
            continue
        if name in ("k_cache", "v_cache") and layout == "xvec":
            P, H, Dx, BS, x = t.shape
            t = t.permute(0, 3, 1, 2, 4).reshape(P, BS, H, Dx * x)
        t = t.cpu().contiguous()
        if t.element_size() == 2:
            d[name] = t.view(torch.int16).numpy().view(np.uint16)
        elif t.dtype in (torch.int8, torch.float32):
            d[name] = t.numpy()
        else:
            d[name] = t.view(torch.uint8).numpy()
    return d


def snapshot_timed_step(st):
    """Replay the timed step graph once more (out poisoned with NaN first)
    and copy its inputs, its output and the cache it leaves to the host.
    Uses no oracle."""
    w = st.w
    st.out.fill_(float("nan"))
    st.replay_step()
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0, "device error flag %d" % int(st.err.item())

    def h(t):
        return None if t is None else t.cpu()
    hw = dataclasses.replace(
        w, context_lens=h(w.context_lens), block_tables=h(w.block_tables), q=h(w.q),
        new_req=h(w.new_req), new_pos=h(w.new_pos), k_new=h(w.k_new), v_new=h(w.v_new),
        k_scale=h(w.k_scale), v_scale=h(w.v_scale), k_block_scale=h(w.k_block_scale),
        v_block_scale=h(w.v_block_scale), k_new_scale=h(w.k_new_scale),
        v_new_scale=h(w.v_new_scale), k_cache0=None, v_cache0=None, fill_req=None,
        fill_pos=None, k_fill=None, v_fill=None, k_fill_scale=None, v_fill_scale=None)
    return hw, cache_host_logical(st.cache, w.layout), st.out.cpu()


def check_timed_step(snap, orc, nthreads=None, seqs=None):
    """The oracle leg's check of a timed step (snapshot_timed_step):
    the oracle re-applies the step's append (its own slot mapping and
    quantisation) to a copy of the GPU's cache, which must leave every byte
    unchanged, and decodes every (sequence, head) over the GPU's cache; the
    largest absolute error of the GPU's output against it is compared with
    the stated tolerance (4e-3 fp16 outputs, 2e-2 bf16)."""
    from tests import pipeline as PL
    hw, c, out = snap
    t0 = time.perf_counter()
    c2 = {k: v.copy() for k, v in c.items()}
    mode = {"head": orc.SCALE_PER_HEAD, "block": orc.SCALE_PER_BLOCK,
            "token": orc.SCALE_PER_TOKEN}[hw.scale_mode]
    req, pos = hw.new_req.numpy(), hw.new_pos.numpy()
    slots = orc.build_slot_mapping(hw.block_tables.numpy(), req, pos, hw.block_size)
    bad = orc.kv_append(PL.KIND_CODE_ORACLE[hw.cache_kind], PL.src_code(hw), W.bits16(hw.k_new),
                        W.bits16(hw.v_new), slots, c2["k_cache"], c2["v_cache"],
                        None if hw.k_scale is None else hw.k_scale.numpy(),
                        None if hw.v_scale is None else hw.v_scale.numpy(), c2.get("k_qscale"),
                        c2.get("k_qzero"), c2.get("v_qscale"), c2.get("v_qzero"),
                        scale_mode=mode,
                        k_new_scale=None if hw.k_new_scale is None else hw.k_new_scale.numpy(),
                        v_new_scale=None if hw.v_new_scale is None else hw.v_new_scale.numpy(),
                        k_scales=c2.get("k_scales"), v_scales=c2.get("v_scales"))
    append_exact = bad == 0 and all(np.array_equal(c[k], c2[k]) for k in c)
    del c2
    Hq = hw.num_heads
    if seqs is None:
        seqs = list(range(hw.batch))
    pairs = np.concatenate([np.arange(b * Hq, (b + 1) * Hq) for b in seqs]).astype(np.int32)
    ref = PL.oracle_decode(hw, orc, c, pairs=pairs, nthreads=nthreads)[seqs]
    got = out.to(torch.float64).numpy()[seqs]
    finite = bool(np.isfinite(got).all())
    max_abs = float(np.abs(got - ref).max()) if finite else float("inf")
    tol = PL.tolerance(hw)
    return {"rows": int(got.shape[0] * got.shape[1]), "of_rows": hw.batch * Hq,
            "max_abs": max_abs, "tolerance": tol,
            "ok": bool(finite and max_abs <= tol and append_exact),
            "append_bit_exact": bool(append_exact), "oracle_s": round(time.perf_counter() - t0, 2),
            "what": "%s of the timed step's output vs the fp64 oracle over the cache the "
                    "step left; the step's appended rows re-applied by the oracle change no "
                    "byte" % ("every (sequence, head)" if len(seqs) == hw.batch else
                             "every head of sequences %s" % seqs)}


# ---------------------------------------------------------------- oracle arms

class OracleArm:
    """The CPU oracle on a bounded sample of a workload: the first sequences
    whose decode fits in about ``budget_s`` seconds on the host cores.  The
    sample's caches are built once (untimed); a timed step is the oracle's
    append of the step's new tokens for those sequences plus their decode
    (all heads)."""

    def __init__(self, w_host, orc, budget_s=15.0, nthreads=None):
        from tests import pipeline as PL
        self.PL, self.w, self.orc = PL, w_host, orc
        self.nthreads = orc.max_threads() if nthreads is None else nthreads
        w = w_host
        if w.q is None:                     # append-only workload
            self.seqs = list(range(w.batch))
        else:
            # rate probe: one sequence, 16-bit reading of its cost
            ctx = w.context_lens.to(torch.int64).numpy()
            probe = [int(np.argmin(ctx))]
            c = PL.oracle_caches(w, orc, seqs=probe)
            pairs = np.arange(probe[0] * w.num_heads, (probe[0] + 1) * w.num_heads,
                              dtype=np.int32)
            t0 = time.perf_counter()
            PL.oracle_decode(w, orc, c, pairs=pairs, nthreads=self.nthreads)
            rate = ctx[probe[0]] / max(1e-6, time.perf_counter() - t0)   # tokens/s, all heads
            budget_tokens = rate * budget_s
            self.seqs, acc = [], 0
            for b in range(w.batch):
                if self.seqs and acc + ctx[b] > budget_tokens:
                    break
                self.seqs.append(b)
                acc += int(ctx[b])
        self.cache = PL.oracle_caches(w, orc, seqs=self.seqs)
        self.pairs = None
        if w.q is not None:
            self.pairs = np.concatenate([np.arange(b * w.num_heads, (b + 1) * w.num_heads)
                                         for b in self.seqs]).astype(np.int32)
        self.bytes = self._bytes()

    def _bytes(self):
        w = self.w
        D, Hkv, BS = w.head_dim, w.num_kv_heads, w.block_size
        row = {"f16": 2 * D, "bf16": 2 * D, "e4m3": D, "e5m2": D, "i8": D, "u3": 3 * D // 8}[w.cache_kind]
        meta = 3 if w.cache_kind == "u3" else 0
        req = w.new_req.numpy()
        sel = np.isin(req, self.seqs) & (w.new_pos.numpy() >= 0)
        n = int(sel.sum())
        total = n * Hkv * 2 * (2 * D + row + meta) + 16 * n
        if w.q is not None:
            for b in self.seqs:
                ctx = int(w.context_lens[b])
                total += ctx * Hkv * 2 * (row + meta) + 4 * w.num_heads * D
                total += (ctx + BS - 1) // BS * 4 + 4
        return total

    def step(self):
        w, PL, orc = self.w, self.PL, self.orc
        t0 = time.perf_counter()
        req = w.new_req.numpy()
        idx = np.nonzero(np.isin(req, self.seqs) & (w.new_pos.numpy() >= 0))[0]
        slots = orc.build_slot_mapping(w.block_tables.numpy(), req[idx], w.new_pos.numpy()[idx],
                                       w.block_size)
        c = self.cache
        ti = torch.from_numpy(idx)
        orc.kv_append(PL.KIND_CODE_ORACLE[w.cache_kind], PL.src_code(w),
                      W.bits16(w.k_new[ti]), W.bits16(w.v_new[ti]), slots, c["k_cache"],
                      c["v_cache"], None if w.k_scale is None else w.k_scale.numpy(),
                      None if w.v_scale is None else w.v_scale.numpy(), c.get("k_qscale"),
                      c.get("k_qzero"), c.get("v_qscale"), c.get("v_qzero"))
        if w.q is not None:
            PL.oracle_decode(w, orc, c, pairs=self.pairs, nthreads=self.nthreads)
        return self.bytes, time.perf_counter() - t0

    def describe(self, seconds):
        w = self.w
        what = ("append of the step's tokens + decode (all heads) of %d/%d sequences"
                % (len(self.seqs), w.batch)) if w.q is not None else (
            "append of all %d tokens" % w.new_req.shape[0])
        return "%s, %d threads, %.2f s per sample" % (what, self.nthreads, seconds)


# ---------------------------------------------------------------- main

def run_reference(args, ws, rank):
    """The reference arm: the CPU oracle, timed as it stands."""
    if rank != 0:
        return 0
    import oracle as orc
    orc.build()
    w = make_workload(args.workload, "cpu")
    per_step = max(1.0, min(15.0, 120.0 / max(1, args.steps + args.warmup)))
    arm = OracleArm(w, orc, budget_s=per_step)
    times, nbytes_all = [], []
    for i in range(args.warmup + args.steps):
        nb, sec = arm.step()
        if i >= args.warmup:
            times.append(sec)
            nbytes_all.append(nb)
    threads, desc = arm.nthreads, arm.describe(float(np.mean(times)))
    value = sum(nbytes_all) / sum(times) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * sum(times) / len(times), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args.workload, ws),
            "device": "host cores",
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


METRIC = "paged-decode effective HBM GB/s (% of GB300 peak); KV append tokens/s"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="fp8_long")
    ap.add_argument("--extra", default="gqa_bf16,u3_mha,mixed_append,mha_short,fp8_long_e5m2,i8_long,"
                                       "fp8_long_token_scales,fp8_long_block_scales,gqa_bf16_xvec,"
                                       "fp8_long_xvec,fp8_long_g16,gqa_bf16_g16,fp8_long_d64,u3_g8,u3_g16",
                    help="other workloads measured in the same run ('' for none)")
    ap.add_argument("--extra-steps", type=int, default=200)
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-splits", type=int, default=0,
                    help="explicit split count for every decode call (> 0 selects the general "
                         "kernel; 0: the automatic plan)")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    ws, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, ws, rank)

    import paged_kv_cache_num_gb300 as pkv
    pkv.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    peak, peak_src = measured_peaks()
    flush = L2Flush(dev)

    # ---------------- main workload, device-timed
    w = make_workload(args.workload, dev, rank)
    step_bytes = algorithmic_bytes(w)
    dec_bytes = algorithmic_bytes(w, append=False)
    app_bytes = algorithmic_bytes(w, decode=False)
    n_real = int((w.new_pos >= 0).sum())
    st = Step(w, pkv, args.num_splits)
    fill = None
    if st.fill is not None:
        fg = st.fill["bytes"] / (st.fill["ms"] * 1e-3) / 1e9
        fill = {"tokens": st.fill["tokens"], "ms": round(st.fill["ms"], 4), "gbs": round(fg, 1),
                "frac_of_peak": round(fg / peak, 4),
                "what": "one context-fill append launch (slots given), CUDA events, best of 3"}
    st.capture()
    for _ in range(args.warmup):
        flush.zero_()
        st.replay_step()
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        tot, _, _ = time_steps(st, args.steps, 0, flush, parts=False)
        wall = time.perf_counter() - t0
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    ms_max, value = job_throughput(pg, step_bytes, float(np.mean(tot)), dev)
    # the step's parts, each replayed alone (outside the timed region)
    nparts = min(args.steps, 500)
    app = time_graph(st.replay_append, nparts, flush)
    dec = time_graph(st.replay_decode, nparts, flush)
    dec_ms = float(np.mean(dec))
    app_ms = float(np.mean(app))
    assert int(st.err.item()) == 0, "device error flag %d" % int(st.err.item())
    check_oracle = rank == 0 and not args.no_cpu_baseline
    snap = snapshot_timed_step(st) if check_oracle and w.q is not None else None

    # ---------------- e2e through the public API with host buffers
    # the step's inputs packed into one pinned host buffer (256-byte aligned
    # sub-buffers), moved by one host-to-device copy per step
    names = ("q", "k_new", "v_new", "new_req", "new_pos", "block_tables", "context_lens")
    src = {k: getattr(w, k).contiguous() for k in names}
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += (src[k].numel() * src[k].element_size() + 255) // 256 * 256
    hpack = torch.empty(total, dtype=torch.uint8).pin_memory()
    dpack = torch.empty(total, dtype=torch.uint8, device=dev)

    def view(buf, k):
        t = src[k]
        n = t.numel() * t.element_size()
        return buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
    for k in names:
        view(hpack, k).copy_(src[k].cpu())
    dbuf = {k: view(dpack, k) for k in names}
    out_host = torch.empty(w.q.shape, dtype=w.q.dtype).pin_memory()
    h2d = total                         # bytes the one copy moves (with alignment gaps)
    d2h = out_host.numel() * out_host.element_size()
    s = torch.cuda.current_stream()

    def e2e_once():
        dpack.copy_(hpack, non_blocking=True)
        if st.fused:
            pkv.decode_step(dbuf["k_new"], dbuf["v_new"], dbuf["new_req"], dbuf["new_pos"],
                            dbuf["q"], st.cache, dbuf["block_tables"], dbuf["context_lens"],
                            sm_scale=w.sm_scale, out=st.out, slots=st.slots,
                            num_splits=st.num_splits, workspace=st.ws, err_flag=st.err)
        else:       # per-token scales: the separate calls (see Step.run)
            st.append(dbuf["new_req"], dbuf["new_pos"], dbuf["k_new"], dbuf["v_new"])
            st.decode(dbuf["q"])
        out_host.copy_(st.out, non_blocking=True)

    def e2e_times(run):
        t = []
        for i in range(args.e2e_steps + 3):
            flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            run()
            s.synchronize()
            if i >= 3:
                t.append(time.perf_counter() - t0)
        return 1e3 * float(np.mean(t))
    # eager: each step calls the API from Python
    e2e_eager_ms, e2e_eager_val = job_throughput(pg, step_bytes, e2e_times(e2e_once), dev)
    # graph: the same calls (pinned host-to-device copy, pkv_decode_step,
    # device-to-host copy) captured once and replayed each step, as a
    # serving loop would; the copies still move the host data every step
    e2e_once()
    torch.cuda.synchronize()
    g_e2e = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(s)
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g_e2e, stream=cs):
            e2e_once()
    s.wait_stream(cs)
    torch.cuda.synchronize()
    e2e_ms, e2e_val = job_throughput(pg, step_bytes, e2e_times(g_e2e.replay), dev)

    # ---------------- roofline of the dominant operation (paged_decode)
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    roofline = decode_roofline(args.workload, dec_bytes, dec_ms, peak, peak_src, args.num_splits)

    # copy-kernel yardstick (1 GiB each way)
    a = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    b = torch.empty_like(a)
    for _ in range(3):
        pkv.copy_peak(a, b)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(10):
        pkv.copy_peak(a, b)
    e1.record()
    torch.cuda.synchronize()
    copy_gbs = 2 * a.numel() * 10 / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del a, b

    # ---------------- other workloads (device-timed, same protocol)
    extra = {}
    launches_per_step = st.launches
    del st
    torch.cuda.empty_cache()
    for name in [x for x in args.extra.split(",") if x]:
        wx = make_workload(name, dev, rank)
        sb = algorithmic_bytes(wx)
        db = algorithmic_bytes(wx, append=False)
        ab = algorithmic_bytes(wx, decode=False)
        nr = int((wx.new_pos >= 0).sum())
        sx = Step(wx, pkv, args.num_splits)
        tt, aa, dd = time_steps(sx, args.extra_steps, max(3, args.warmup // 4), flush)
        assert int(sx.err.item()) == 0, name
        e = {"step_ms": round(float(np.mean(tt)), 4),
             "append_tokens_per_s": round(nr / (float(np.mean(aa)) * 1e-3), 1),
             "append_gbs": round(ab / (float(np.mean(aa)) * 1e-3) / 1e9, 1)}
        if wx.q is not None:
            g = db / (float(np.mean(dd)) * 1e-3) / 1e9
            e.update({"decode_ms": round(float(np.mean(dd)), 4), "decode_gbs": round(g, 1),
                      "decode_frac_of_peak": round(g / peak, 4),
                      "decode_algorithmic_bytes": db,
                      "roofline": decode_roofline(name, db, float(np.mean(dd)), peak, peak_src,
                                                  args.num_splits)})
            if check_oracle:
                import oracle as orc
                orc.build()
                # the first and the last sequence, all heads (the headline
                # workload's check covers every sequence)
                e["parity"] = check_timed_step(snapshot_timed_step(sx), orc,
                                               seqs=sorted({0, wx.batch - 1}))
        if sx.fill is not None:
            fg = sx.fill["bytes"] / (sx.fill["ms"] * 1e-3) / 1e9
            e["fill_append"] = {"tokens": sx.fill["tokens"], "ms": round(sx.fill["ms"], 4),
                                "gbs": round(fg, 1), "frac_of_peak": round(fg / peak, 4),
                                "what": "one context-fill append launch (slots given), "
                                        "CUDA events, best of 3"}
        extra[name] = e
        del sx, wx
        torch.cuda.empty_cache()

    if rank == 0:
        extra["pack3_2^24"] = time_pack3_bijection(pkv, dev, flush)
        torch.cuda.empty_cache()

    # ---------------- CPU oracle on a bounded sample
    cpu = parity = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle as orc
        orc.build()
        wh = make_workload(args.workload, "cpu")
        arm = OracleArm(wh, orc, budget_s=10.0)
        nb, sec = arm.step()
        cpu = {"value": round(nb / sec / 1e9, 4), "unit": "GB/s", "cores": arm.nthreads,
               "kind": "oracle", "sample": arm.describe(sec)}
        del arm
        # a smaller sample of the same workload on one host core
        arm = OracleArm(wh, orc, budget_s=4.0, nthreads=1)
        nb1, sec1 = arm.step()
        cpu["single_thread"] = {"value": round(nb1 / sec1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                                "sample": arm.describe(sec1)}
        del arm, wh
        # the oracle's 2^24-octet pack + unpack (one thread), beside the pages' CPU time
        vals = W.all_octets("cpu").numpy().reshape(-1, 8)
        t0 = time.perf_counter()
        packed = orc.pack3(vals)
        back = orc.unpack3(packed)
        t_or = time.perf_counter() - t0
        if "pack3_2^24" in extra:
            extra["pack3_2^24"]["oracle_pack_unpack_s"] = round(t_or, 3)
            extra["pack3_2^24"]["oracle_roundtrip_ok"] = bool(np.array_equal(back, vals))
        del vals, packed, back
        # the timed step's own output and cache, checked by the oracle
        if snap is not None:
            parity = check_timed_step(snap, orc)
            del snap

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.cache_kind,
            "data": "synthetic (seeded torch CUDA generator; N(0,1) K/V/q)",
            "config": workload_config(w, args.workload, ws),
            "timing": {"num_splits": args.num_splits, "l2": "inputs larger than L2, and flushed between steps outside the "
                             "timed events (256 MiB write, then a 512 MiB read that drains "
                             "its write-back)",
                       "launch": "a device-timed step replays one CUDA graph of one "
                                 "pkv_decode_step call (append kernel with the slot "
                                 "computation fused, decode, merge; programmatic dependent "
                                 "launches); its append (pkv_slot_mapping + pkv_kv_append) and "
                                 "decode parts are replayed alone for the breakdown; e2e "
                                 "replays one graph of [one packed "
                                 "host-to-device copy of the step's inputs, pkv_decode_step "
                                 "(slot mapping, append, decode), the device-to-host copy of "
                                 "out] per step (e2e_eager: the same calls made eagerly)"},
            "pct_of_peak": round(100 * value / peak, 2),
            "decode_gbs": round(dec_gbs, 1), "decode_ms": round(dec_ms, 5),
            "append_tokens_per_s": round(n_real / (app_ms * 1e-3), 1),
            "append_ms": round(app_ms, 5),
            "fill_append": fill,
            "step_algorithmic_bytes": step_bytes,
            "roofline": roofline,
            "copy_kernel_gbs": round(copy_gbs, 1),
            "clocks": clk.summary(),
            "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                    "how": "host wall clock per step around one CUDA-graph replay of [pinned "
                           "host-to-device copy of the step's inputs, pkv_decode_step, "
                           "device-to-host copy of out] and a stream synchronize"},
            "e2e_eager": {"value": round(e2e_eager_val, 2), "unit": "GB/s",
                          "ms_per_step": round(e2e_eager_ms, 4),
                          "how": "the same calls made eagerly from Python each step"},
            "gpu_launches": launches_per_step * args.steps,
            "cpu_baseline": cpu,
            "parity": parity,
            "workloads": extra,
            "timed_wall_s": round(wall, 3),
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
