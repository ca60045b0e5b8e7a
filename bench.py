"""Benchmark of the KATA chunked forward on GB300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one kata_fwd_chunked call over one batch of the workload (the
feature lift, intra-chunk term, chunk state, inter-chunk prefix scan and the
normalised output, all inside the call).  Inputs are resident in HBM before
the timed region and are larger than L2 (129 MB) for the default workload, so
no L2 flush is needed; the timed region is K back-to-back steps bracketed by a
barrier and torch.cuda.synchronize(), timed with CUDA events on the launching
stream, max over ranks.  Workloads whose inputs fit in L2 write a 258 MB buffer
before every step and time each step with its own pair of events.  value = tokens (B*T per step, all heads) per second.

Extra keys: "roofline" for the dominant kernel (its algorithmic work per
launch over its mean CUDA-event launch time, from the library's tracing),
"cpu_baseline" (the CPU oracle on sampled rows of the same workload),
"e2e" (the host-buffer entry point with host<->device copies in the timed
region), "decode" (the recurrent decode step at batch 256), "clocks"
(nvidia-smi samples during the timed region) and "gpu_launches".

--impl reference times the CPU oracle (the reference implementation of this
repository; there is no installable upstream code) on bounded row samples of
the same workload.  Multi-GPU runs are independent replicas (the path shards
over (b, h) with no exchange), scaling "weak".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

DEFAULT_WORKLOAD = "long_ctx_bf16"
L2_BYTES = 129 * 1024 * 1024
SMS = 152
FP32_FFMA_PEAK_TFLOPS = SMS * 128 * 2 * 2.070e9 / 1e12   # 152 SMs x 128 lanes x FMA x 2.07 GHz


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------------------
# algorithmic work per launch of each kernel (stated in the design notes)


def _intra_pairs(T, C):
    """Causal (s <= t) pairs inside chunks, summed over the chunks of one head."""
    full, tail = divmod(T, C)
    return full * C * (C + 1) // 2 + tail * (tail + 1) // 2


def tc_plan(w, num_sms: int):
    """Segmentation of the d = 32 tensor path for workload w, as the library
    reports it (kata_fwd_segments): 128-token chunks, G segments of Lc chunks per
    head.  num_sms is the device's, which the library reads itself."""
    nct = -(-w.T // 128)
    import kernelized_causal_linear_gb300 as kg
    G, seg_tokens = kg.kata_fwd_segments(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype)
    return nct, G, max(1, seg_tokens // 128)


class FeatureMap:
    """The forward's feature map: the full rank-one map or a reduced PSD family
    ([KATA] Sec. 4.1) with g blocks; the Sigma maps take the eps and scale of the
    pages' Sigma configuration (eps = 1e-4; scale 1/4 for Sigma_4, else 1)."""
    CODES = {"full": 0, "M": 1, "Sigma": 2, "orthant": 3}

    def __init__(self, name: str = "full", g: int = 1):
        self.name, self.g, self.code = name, int(g), self.CODES[name]
        self.eps = 1e-4 if name == "Sigma" else 1e-6 if name == "orthant" else 0.0
        self.scale = (0.25 if self.g == 4 else 1.0) if name == "Sigma" else 1.0

    def n(self, d: int) -> int:
        m = d // self.g
        return {0: d * (d + 1) // 2, 1: self.g * m * (m + 1) // 2, 2: m * (m + 1) // 2,
                3: d}[self.code]

    def intra_d(self, d: int) -> int:
        """Multiply-adds per (t, s) pair of the closed-form weight: all g x g block
        products for Sigma_g, d otherwise."""
        return self.g * d if self.code == 2 else d

    def label(self) -> str:
        return {0: "full", 3: "orthant"}.get(self.code, f"{self.name}_{self.g}")


FULL_MAP = FeatureMap()


def stage_work(stage: str, w, num_sms: int = SMS, fm: FeatureMap = FULL_MAP):
    """(algorithmic work per launch, unit, bound) for a traced stage on workload w."""
    BH, T, d, dv, C, n = w.B * w.H, w.T, w.d, w.dv, w.C, fm.n(w.d)
    NC = -(-T // C)
    state_flops = 2.0 * n * (dv + 1) * T * BH          # Psi(K)^T [V|1]
    out_inter = 2.0 * n * (dv + 1) * T * BH            # Psi(Q) [S|Z]
    intra = 2.0 * (fm.intra_d(d) + dv + 1) * _intra_pairs(T, C) * BH   # weights and P [V|1], causal
    if stage == "simt_chunk_state":
        return state_flops, "TFLOP/s", "alu"
    if stage == "simt_output":
        return out_inter + intra, "TFLOP/s", "alu"
    if stage == "simt_scan":
        return 2.0 * 4 * n * (dv + 1) * NC * BH, "GB/s", "hbm"
    if stage == "simt_scan_blocked":   # the records are read twice, written once
        return 3.0 * 4 * n * (dv + 1) * NC * BH, "GB/s", "hbm"
    # GatedKATA on CUDA cores: the same contractions (the gate products add O(C)
    # multiplies per chunk); the gated scan also reads one gate product per chunk
    if stage == "gated_chunk_state":
        return state_flops, "TFLOP/s", "alu"
    if stage == "gated_output":
        return out_inter + intra, "TFLOP/s", "alu"
    if stage == "gated_scan":
        return (2.0 * 4 * n * (dv + 1) + 4) * NC * BH, "GB/s", "hbm"
    if stage.startswith("tc_"):
        nct, G, Lc = tc_plan(w, num_sms)
        seg_tokens = min(T, (G - 1) * Lc * 128) * BH      # tokens in all but the last segments
        if stage == "tc_segment_state":
            return 2.0 * n * (dv + 1) * seg_tokens, "TFLOP/s", "tensor"
        # GatedKATA on the tensor path: the same contractions as the plain kernels;
        # the piece prep reads and writes the scaled keys of the summed segments,
        # the gated scan reads and writes the records with one multiplier each
        if stage == "tc_gated_piece_prep":
            return 2.0 * 2 * d * seg_tokens + 4.0 * nct * BH, "GB/s", "hbm"
        if stage == "tc_gated_scan":
            rec = 4.0 * (5 * 128 * dv + d * d)
            return 2.0 * rec * G * BH, "GB/s", "hbm"
        if stage in ("tc_segment_output", "tc_pair_output", "tc_segment_output_gated"):
            intra128 = 2.0 * (fm.intra_d(d) + dv + 1) * _intra_pairs(T, 128) * BH
            return state_flops + out_inter + intra128, "TFLOP/s", "tensor"
        if stage == "tc_segment_scan":
            rec = 4.0 * (5 * 128 * dv + d * d)
            return 2.0 * rec * G * BH, "GB/s", "hbm"
    if stage == "tc_gate_prep":
        # reads k and the gates, writes the scaled keys and the cumulative log2 gates
        return float(BH * T) * (2 * d * 2 + 2 * 4), "GB/s", "hbm"
    if stage in ("tc_quadratic", "tc_quadratic_gated"):
        # every causal (t, s <= t) pair of the head: (q.k)^2 and P [V|1]
        return 2.0 * (d + dv + 1) * _intra_pairs(T, T) * BH, "TFLOP/s", "tensor"
    if stage == "tc_sub_finalize":
        # M_2 / M_4 sub-heads: reads their fp32 numerators and denominators, writes bf16 out
        nsub = 4 if (fm.code, fm.g) == (1, 4) else 2
        return float(BH * T) * (nsub * (dv + 1) * 4 + dv * 2), "GB/s", "hbm"
    if stage == "tc_m4_pad":
        # q and k rows in, zero-padded to four 32-wide blocks out
        return float(BH * T) * 2 * (d * 2 + 4 * 32 * 2), "GB/s", "hbm"
    # Sigma_g finalize: 128-token chunk sums of v, |k|^2 v, |k|^2 (reads k, v, writes
    # one record per chunk), their exclusive scan, and the pass that reads the fp32
    # partial numerators and denominators with q, k, v and writes bf16 out: four of
    # each for Sigma_2 (crosswise sub-heads), four numerators (feature groups) and one
    # denominator for Sigma_1 at d = 64, one of each for Sigma_1 at d = 32
    rec_sigma = 4.0 * (2 * dv + 4)
    nn, nd = (1, 1) if (fm.g == 1 and d == 32) else (4, 1) if fm.g == 1 else (4, 4)
    if stage == "tc_sigma_sums":
        return float(BH * T) * (d + dv) * 2 + rec_sigma * -(-T // 128) * BH, "GB/s", "hbm"
    if stage == "tc_sigma_scan":
        return 2.0 * rec_sigma * -(-T // 128) * BH, "GB/s", "hbm"
    if stage == "tc_sigma_finalize":
        return (float(BH * T) * ((nn * dv + nd) * 4 + (2 * d + dv) * 2 + dv * 2)
                + rec_sigma * -(-T // 128) * BH), "GB/s", "hbm"
    if stage == "tc64_output":
        intra128 = 2.0 * (d + dv + 1) * _intra_pairs(T, 128) * BH
        return state_flops + out_inter + intra128, "TFLOP/s", "tensor"
    if stage == "tc64_finalize":
        # reads four fp32 partial numerators and the denominator, writes bf16 out
        return float(BH * T) * (4 * dv * 4 + 4 + dv * 2), "GB/s", "hbm"
    # explicit-feature tensor path (reduced maps with few features): the lift reads
    # q or k and writes its features (n rounded up to 8, bf16), the state kernel
    # forms Phi_K^T V per chunk (tensor) and writes an fp32 record [n][65], the scan
    # reads and writes the records, the output kernel forms Phi_Q Phi_K^T, Phi_Q
    # S_pre and P V (tensor; algorithmic: the inter term and the causal pairs)
    if stage == "tc_feat_lift":
        return float(BH * T) * (d * 2 + ((n + 7) // 8 * 8) * 2), "GB/s", "hbm"
    if stage == "tc_feat_state":
        return 2.0 * n * dv * T * BH, "TFLOP/s", "tensor"
    if stage == "tc_feat_scan":
        return 2.0 * 4 * n * (dv + 1) * -(-T // 128) * BH, "GB/s", "hbm"
    if stage == "tc_feat_output":
        return (2.0 * n * (dv + 1) * T * BH +
                2.0 * (n + dv + 1) * _intra_pairs(T, 128) * BH), "TFLOP/s", "tensor"
    # other bf16 head sizes on the tensor kernels: q or k padded to 32 columns
    # (one launch each), v cut into 64-column parts, each part's output columns
    # copied out, each part's state gathered (w: the v columns of one part)
    wp = min(dv, 64)
    if stage == "tc_adapt_pad":
        return float(BH * T) * (d * 2 + 32 * 2), "GB/s", "hbm"
    if stage == "tc_adapt_v_part":
        return float(BH * T) * (wp * 2 + 64 * 2), "GB/s", "hbm"
    if stage == "tc_adapt_out_part":
        return float(BH * T) * (wp * 2 + wp * 2), "GB/s", "hbm"
    if stage == "tc_adapt_state_part":
        return float(BH) * n * (wp + 1) * 4 * 2, "GB/s", "hbm"
    return None, "", ""


def kernel_workload(w, path):
    """The shape the tensor-core kernels run for w: a bf16 head with d = 16 or
    dv != 64 runs on them with q, k padded to d = 32 and v cut into 64-column
    parts (one launch of each kernel per part), so their per-launch work is that
    of the padded shape with dv = 64."""
    if path != 2 or w.dtype != torch.bfloat16 or (w.d != 16 and w.dv == 64):
        return w
    return w.scaled(d=max(w.d, 32), dv=64)


def stage_dense_flops(stage: str, w, num_sms: int = SMS, fm: FeatureMap = FULL_MAP):
    """Tile-level flops a tensor-core launch executes (padding and masked halves
    included), for the kernels whose MMA tiles are fixed: per 128-token chunk the
    d = 32 output kernel runs 5 state blocks (M128 N64 K128), psi_q S_pre over 4
    full blocks and one 16-feature block, 4 Q K^T quarters (M128 N32 K32), 4 P V
    quarters (M128 N64 K32), the Gram (M128 N32 K128) and Q G_pre (M128 N32 K32);
    the state kernel the 5 state blocks and the Gram.  The quadratic kernels run
    every (query tile, key tile <= it) pair as full 128 x 128 tiles.  The reduced
    maps on the tensor path run d = 32 sub-heads: 2 per head for M_2, 4 for
    M_4 (zero-padded blocks) and Sigma_2 (whose segment sums need only the 2 key
    halves)."""
    BH, T, d, dv = w.B * w.H, w.T, w.d, w.dv
    if d == 64 and (fm.code, fm.g) in ((1, 2), (2, 2), (1, 4)):
        sub_w = w.scaled(B=w.B * (2 if (fm.code, fm.g) == (1, 2) else 4), d=32)
        if stage == "tc_segment_state" and fm.code == 2:
            sub_w = w.scaled(B=w.B * 2, d=32)
        return stage_dense_flops(stage, sub_w, num_sms)
    mma = lambda m, n, k: 2.0 * m * n * k
    nct, G, Lc = tc_plan(w, num_sms)
    state = 5 * mma(128, 64, 128)
    gram = mma(128, 32, 128)
    if stage in ("tc_segment_output", "tc_segment_output_gated"):
        per = (state + 4 * mma(128, 64, 128) + mma(128, 64, 16) + 4 * mma(128, 32, 32)
               + 4 * mma(128, 64, 32) + gram + mma(128, 32, 32))
        return per * nct * BH
    if stage == "tc_pair_output":
        # over the CTA pair: the 5 state blocks, psi_q S_pre over 4 full blocks and
        # the 32-feature block, one Q K^T (M128 N128 K32), P V (M128 N64 K128), the
        # Gram and Q G_pre
        per = (state + 4 * mma(128, 64, 128) + mma(128, 64, 32) + mma(128, 128, 32)
               + mma(128, 64, 128) + gram + mma(128, 32, 32))
        return per * nct * BH
    if stage == "tc_segment_state":
        return (state + gram) * min(nct, (G - 1) * Lc) * BH
    if stage in ("tc_quadratic", "tc_quadratic_gated"):
        nt = -(-T // 128)
        return (nt * (nt + 1) // 2) * BH * (mma(128, 128, d) + mma(128, dv, 128))
    return None


def call_flops(w, fm: FeatureMap = FULL_MAP, algo: str = "chunked") -> float:
    """Algorithmic flops of one forward call at the workload's chunk size:
    2n(dv+1) (state) + 2n(dv+1) (inter output) per token and head, plus the
    causal intra-chunk term 2(d'+dv+1) per (t, s<=t) pair inside chunks (d' the
    weight's multiply-adds: d, or g d for Sigma_g)."""
    BH, T, d, dv, C, n = w.B * w.H, w.T, w.d, w.dv, w.C, fm.n(w.d)
    if algo in ("quadratic", "gated_quadratic"):   # the O(T^2) form: every causal pair
        return 2.0 * (d + dv + 1) * _intra_pairs(T, T) * BH
    return 4.0 * n * (dv + 1) * T * BH + 2.0 * (fm.intra_d(d) + dv + 1) * _intra_pairs(T, C) * BH


# the translation unit of each traced stage's kernel (its launch configuration
# lives there too); every stage also depends on all the shared headers
_STAGE_SOURCE = (("tc_segment", "kata_tc.cu"), ("tc_pair", "kata_tc_pair.cu"),
                 ("tc_gated", "kata_tc.cu"), ("tc_sub_finalize", "kata_tc.cu"),
                 ("tc_m4", "kata_tc.cu"), ("tc_adapt", "kata_adapt.cu"),
                 ("tc_feat", "kata_feat.cu"),
                 ("tc_sigma", "kata_sigma.cu"),
                 ("tc64", "kata_tc64.cu"), ("tc_quadratic", "kata_quad.cu"),
                 ("tc_gate_prep", "kata_quad.cu"), ("simt", "kata_simt.cu"),
                 ("gated", "kata_gated.cu"), ("decode", "kata_decode.cu"))


def _local_includes(path: str, seen: set) -> None:
    """path and, transitively, the quoted local headers it includes."""
    path = os.path.normpath(path)
    if path in seen or not os.path.exists(path):
        return
    seen.add(path)
    with open(path) as f:
        for line in f:
            m = re.match(r'\s*#\s*include\s+"([^"]+)"', line)
            if m:
                _local_includes(os.path.join(os.path.dirname(path), m.group(1)), seen)


def _source_digest(stage: str | None = None) -> str:
    """Digest of the CUDA sources a stage's kernel is built from: its own .cu and
    the local headers it includes, transitively (all of csrc without a stage)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kernelized_causal_linear_gb300", "csrc")
    own = None
    if stage is not None:
        own = next((f for prefix, f in _STAGE_SOURCE if stage.startswith(prefix)), None)
    if own is None:
        files = [os.path.join(csrc, n) for n in os.listdir(csrc) if n.endswith((".cu", ".cuh"))]
    else:
        seen: set = set()
        _local_includes(os.path.join(csrc, own), seen)
        files = list(seen)
    for path in sorted(files, key=lambda x: os.path.relpath(x, ROOT)):
        with open(path, "rb") as f:
            h.update(os.path.relpath(path, ROOT).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def _ncu_traffic(kernel_stage: str, workload: str):
    """DRAM bytes per launch for a stage from the committed ncu summary, if it
    was taken on the current sources of that stage's kernel; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    digest = _source_digest(kernel_stage)
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 4 and not line.startswith("#"):
                stage, wl, sha, nbytes = parts
                if stage == kernel_stage and wl == workload and sha == digest:
                    return float(nbytes)
    return None


# ----------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    """nvidia-smi clocks/throttle samples every 5 ms (about 160 a second on
    GB300, so a 20 ms timed region still holds a few), each stamped with the
    host time it arrived; summary() keeps the samples inside mark_start() ..
    mark_stop() (the timed region)."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.idx = device_index
        self.samples = []
        self.t0 = self.t1 = None

    def _reader(self):
        for line in self.proc.stdout:
            if line.strip():
                self.samples.append((time.time(), line))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "5", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            self.thread = threading.Thread(target=self._reader, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, l in self.samples:
            if self.t0 is not None and not (self.t0 <= ts <= (self.t1 or ts)):
                continue
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# CPU oracle baseline (rank 0 only)


def _oracle_sample(w, q, k, v, seconds: float, rng, fm: FeatureMap = FULL_MAP, gate=None):
    """Time the oracle on sampled output rows (uniform over heads and positions)
    for about `seconds`; returns (rows, elapsed seconds, threads).  Each row is
    one head of one token.  With `gate` ([1, heads, T] fp64) the gated definition."""
    import oracle
    BH = w.B * w.H
    qf = q.reshape(BH, w.T, w.d)
    kf = k.reshape(BH, w.T, w.d)
    vf = v.reshape(BH, w.T, w.dv)
    gf = gate.reshape(BH, w.T) if gate is not None else None

    def run(nrows):
        heads = rng.integers(0, BH, size=nrows)
        ts = rng.integers(0, w.T, size=nrows)
        t0 = time.perf_counter()
        for h in np.unique(heads):
            sel = ts[heads == h]
            if gf is not None:
                oracle.forward_rows_gated(qf[h][None, None], kf[h][None, None], vf[h][None, None],
                                          gf[h][None, None], sel)
            elif fm.code == 0:
                oracle.forward_rows(qf[h][None, None], kf[h][None, None], vf[h][None, None], sel)
            else:
                oracle.forward_rows_map(qf[h][None, None], kf[h][None, None], vf[h][None, None],
                                        sel, fm.name, fm.g, fm.eps, fm.scale)
        return time.perf_counter() - t0

    probe = 16
    dt = run(probe)
    while dt < min(1.0, seconds / 4):          # calibrate on at least ~1 s of work
        probe *= 4
        dt = run(probe)
    nrows = max(probe, int(probe * seconds / dt))
    dt = run(nrows)
    return nrows, dt, oracle.get_threads()


def _cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        fields = dict(line.split(":", 1) for line in out.splitlines() if ":" in line)
        for key in ("Model name", "Vendor ID"):
            name = fields.get(key, "").strip()
            if name and name != "-":
                return name
    except (OSError, subprocess.SubprocessError, ValueError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part", "hardware")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def _cpu_extras(w, qh, kh, vh, seconds: float, fm: FeatureMap, gate):
    """More CPU reference points: the same sampled direct oracle on one core, and
    the O(T n dv) feature-state recurrence (the fairer CPU algorithm) on a prefix of
    each kept head (its cost per token is the same at every position)."""
    import oracle
    extras = {"cpu_model": _cpu_model(), "nproc": os.cpu_count()}
    prev = oracle.get_threads()
    oracle.set_threads(1)
    try:
        nrows, dt, _ = _oracle_sample(w, qh, kh, vh, max(1.0, seconds / 3),
                                      np.random.default_rng(2), fm, gate)
        extras["single_core"] = {"value": (nrows / w.H) / dt, "unit": "tokens/s", "cores": 1,
                                 "sample": f"{nrows} output rows, direct O(T^2) fp64, {dt:.1f} s"}
    finally:
        oracle.set_threads(prev)
    if fm.code == 0 and gate is None:
        heads = qh.shape[1]
        L = min(w.T, 256)
        while True:   # a prefix of L tokens on every kept head, about seconds / 3 of work
            t0 = time.perf_counter()
            oracle.recurrent(qh[:, :, :L], kh[:, :, :L], vh[:, :, :L])
            dt = time.perf_counter() - t0
            if dt >= max(0.5, seconds / 6) or L >= w.T:
                break
            L = min(w.T, L * 4)
        extras["recurrent_form"] = {
            "value": (heads * L / w.H) / dt, "unit": "tokens/s",
            "cores": min(heads, oracle.get_threads()), "kind": "oracle recurrence",
            "sample": f"first {L} tokens of heads 0..{heads - 1}, explicit vech-state "
                      f"recurrence (O(T n dv)) in fp64, {dt:.2f} s; tokens = head-tokens / H"}
    return extras


def _host_f64(t):
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def run_reference(args):
    rank = rank_env()[0]
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w = _workload(args)
    fm = FeatureMap(args.map, args.g)
    q, k, v = workloads.make_qkv(w)
    BH = w.B * w.H
    # keep at most 4 heads on the host in fp64 (rows are sampled from them)
    keep = min(BH, 4)
    sub = w.scaled(B=1, H=keep)
    qh = _host_f64(q.reshape(BH, w.T, w.d)[:keep]).reshape(1, keep, w.T, w.d)
    kh = _host_f64(k.reshape(BH, w.T, w.d)[:keep]).reshape(1, keep, w.T, w.d)
    vh = _host_f64(v.reshape(BH, w.T, w.dv)[:keep]).reshape(1, keep, w.T, w.dv)
    gh = None
    if args.algo.startswith("gated"):
        gh = _host_f64(workloads.make_gate(w).reshape(BH, w.T)[:keep]).reshape(1, keep, w.T)
    rng = np.random.default_rng(0)
    per_step_s = float(os.environ.get("KATA_REF_STEP_SECONDS", "3"))
    times, rows_total = [], 0
    for i in range(args.warmup + args.steps):
        nrows, dt, threads = _oracle_sample(sub, qh, kh, vh, per_step_s, rng, fm, gh)
        if i >= args.warmup:
            times.append(dt)
            rows_total += nrows
    # a token of the workload has H heads; each sampled row is one head
    value = (rows_total / w.H) / sum(times)
    line = {
        "impl": "reference", "metric": _metric(), "value": value, "unit": "tokens/s",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(_config(w, fm), algorithm=args.algo),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows_total} output rows of heads 0..{keep - 1}, positions "
                                   f"uniform in [0,T), direct O(T^2) fp64 definition"
                                   f"{' (gated)' if gh is not None else ''}; tokens = rows / H"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _workload(args):
    """The named workload, at --shape B,H,T when given."""
    w = workloads.WORKLOADS[args.workload]
    if args.shape is not None:
        b_, h_, t_ = args.shape
        w = w.scaled(B=b_, H=h_, T=t_)
    if args.head_dims is not None:
        d_, dv_ = args.head_dims
        w = w.scaled(d=d_, dv=dv_)
    return w


def _metric():
    return "fwd tokens/s for chunked PSD linear attention; % bf16 tensor peak (1 GB300)"


def _config(w, fm: FeatureMap = FULL_MAP):
    return {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "dv": w.dv, "C": w.C,
            "feature_map": fm.label(), "feature_dim": fm.n(w.d), "global_batch": w.B,
            "seq_len": w.T,
            "input_dtype": str(w.dtype).replace("torch.", ""),
            "l2": "inputs larger than L2, no flush" if _input_bytes(w) > L2_BYTES
            else "L2 flushed before every step (258 MB write, outside the per-step events)",
            "parallelism": "replicas"}


def _input_bytes(w):
    es = 2 if w.dtype == torch.bfloat16 else 4
    return w.B * w.H * w.T * (2 * w.d + w.dv) * es


# ----------------------------------------------------------------------------


def _dtype_name(w):
    return "bf16" if w.dtype == torch.bfloat16 else "f32"


# ----------------------------------------------------------------------------
# one process per GPU (replicas): rank layout and the whole-job aggregate


def rank_env():
    """(rank, world size, local rank) from the launcher's environment (torchrun
    sets RANK / WORLD_SIZE / LOCAL_RANK; a plain run is rank 0 of 1)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(elapsed_ms: float, dist=None, device="cuda") -> float:
    """The slowest rank's timed region (every rank gets it); no-op on one rank."""
    if dist is None:
        return elapsed_ms
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, elapsed_ms: float) -> float:
    """Whole-job tokens/s: every replica's tokens over the slowest rank's time
    (weak scaling: the per-GPU work stays fixed as ranks are added)."""
    return tokens_per_rank * world / (elapsed_ms / 1e3)


def run_ours(args):
    rank, world, local = rank_env()
    if world != args.gpus:
        if rank == 0:
            sys.stderr.write(f"warning: WORLD_SIZE={world} but --gpus {args.gpus}\n")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from kernelized_causal_linear_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if dist is not None:
        dist.barrier()
    import kernelized_causal_linear_gb300 as kg

    w = _workload(args)
    fm = FeatureMap(args.map, args.g)
    peaks = _peaks()
    q, k, v = workloads.make_qkv(w, device="cuda")
    gate = workloads.make_gate(w, device="cuda") if args.algo.startswith("gated") else None
    out = torch.empty(w.B, w.H, w.T, w.dv, dtype=w.dtype, device="cuda")
    stream = torch.cuda.current_stream()
    if args.algo == "gated_quadratic":
        path = kg.KATA_PATH_TC

        def fwd(q_, k_, v_, out_, g_=gate):
            kg.kata_fwd_quadratic_gated(q_, k_, v_, g_, out=out_)
    elif args.algo == "gated":
        path = kg.kata_fwd_path_gated(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype)

        def fwd(q_, k_, v_, out_, g_=gate):
            kg.kata_fwd_chunked_gated(q_, k_, v_, g_, w.C, out=out_)
    elif args.algo == "quadratic":
        path = kg.KATA_PATH_TC

        def fwd(q_, k_, v_, out_):
            kg.kata_fwd_quadratic(q_, k_, v_, out=out_)
    elif fm.code == 0:
        path = kg.kata_fwd_path(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype)

        def fwd(q_, k_, v_, out_):
            kg.kata_fwd_chunked(q_, k_, v_, w.C, out=out_)
    else:
        path = kg.kata_fwd_path_map(w.B, w.H, w.T, w.d, w.dv, w.C, w.dtype, fm.code, fm.g)

        def fwd(q_, k_, v_, out_):
            kg.kata_fwd_chunked_map(q_, k_, v_, w.C, fm.code, fm.g, fm.eps, fm.scale, out=out_)

    for _ in range(args.warmup):
        fwd(q, k, v, out)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()

    # Inputs smaller than L2: flush L2 before every step by writing a buffer
    # larger than it, and time each step alone (events around the call only).
    flush = None
    if _input_bytes(w) <= L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ev = ([(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)] if flush is not None else [])
    with ClockSampler(torch.cuda.current_device()) as clk:
        time.sleep(0.5)
        kg.kata_trace_begin()
        torch.cuda.synchronize()
        clk.mark_start()
        start.record(stream)
        for i in range(args.steps):
            if flush is not None:
                flush.fill_(i & 0xFF)
                step_ev[i][0].record(stream)
            fwd(q, k, v, out)
            if flush is not None:
                step_ev[i][1].record(stream)
        stop.record(stream)
        torch.cuda.synchronize()
        clk.mark_stop()
        stages = kg.kata_trace_end()
    if dist is not None:
        dist.barrier()
    if flush is not None:
        elapsed_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    else:
        elapsed_ms = start.elapsed_time(stop)
    elapsed_ms = max_over_ranks(elapsed_ms, dist)
    value = job_throughput(w.B * w.T * args.steps, world, elapsed_ms)

    # dominant kernel roofline
    launches = sum(n for n, _ in stages.values())
    dom = max(stages.items(), key=lambda kv: kv[1][1])[0] if stages else None
    roofline = None
    if dom is not None:
        nl, tot = stages[dom]
        wk = w if dom.startswith("tc_adapt") or fm.code != 0 or args.algo != "chunked" \
            else kernel_workload(w, path)
        work, unit, bound = stage_work(dom, wk, torch.cuda.get_device_properties(0).multi_processor_count,
                                       fm)
        mean_s = tot / nl / 1e3
        if work is not None:
            if unit == "TFLOP/s":
                achieved = work / mean_s / 1e12
                if bound == "tensor":
                    peak, psrc = peaks["bf16_tflops"], f"bf16 dense burst, {peaks['source']}"
                else:
                    peak, psrc = FP32_FFMA_PEAK_TFLOPS, "fp32 FFMA: 152 SMs x 128 lanes x 2 x 2.07 GHz"
            else:
                achieved = work / mean_s / 1e9
                peak, psrc = peaks["hbm_gbs"], f"HBM copy, {peaks['source']}"
            traffic = (_ncu_traffic(dom, w.name)
                       if fm.code == 0 and args.shape is None and args.head_dims is None else None)
            roofline = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak,
                        "unit": unit, "frac": achieved / peak, "traffic": traffic,
                        "peak_source": psrc, "mean_launch_ms": mean_s * 1e3,
                        "work_per_launch": work}
            dense = stage_dense_flops(dom, wk, torch.cuda.get_device_properties(0).multi_processor_count,
                                      fm)
            if dense is not None:   # what the tensor cores execute, beside the algorithmic work
                roofline["dense_tflops"] = dense / mean_s / 1e12
                roofline["dense_frac"] = dense / mean_s / 1e12 / peaks["bf16_tflops"]
    # whole-call tensor fraction (algorithmic tensor flops over the step time)
    step_s = elapsed_ms / 1e3 / args.steps
    alg_flops = call_flops(w, fm, args.algo)
    whole = {"algorithmic_tflops": alg_flops / step_s / 1e12,
             "frac_of_bf16_peak": alg_flops / step_s / 1e12 / peaks["bf16_tflops"]}

    # end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e:
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        steps_e2e = max(3, min(args.steps, 10))
        if fm.code == 0 and args.algo == "chunked":   # the C ABI's host-buffer entry point
            def e2e_step():
                kg.kata_fwd_chunked_host(qh, kh, vh, w.C, out=oh)
        else:   # pinned copies in (the gates too), the forward, copy out
            qd, kd, vd, od = (torch.empty_like(t) for t in (q, k, v, out))
            pairs = [(qd, qh), (kd, kh), (vd, vh)]
            if gate is not None:
                gh = gate.cpu().pin_memory()
                gd = torch.empty_like(gate)
                pairs.append((gd, gh))

            def e2e_step():
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
                if gate is not None:
                    fwd(qd, kd, vd, od, gd)
                else:
                    fwd(qd, kd, vd, od)
                oh.copy_(od, non_blocking=True)
                torch.cuda.current_stream().synchronize()
        e2e_step()
        if dist is not None:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(steps_e2e):
            e2e_step()
        dt = max_over_ranks((time.perf_counter() - t0) * 1e3, dist) / 1e3
        es = qh.element_size()
        gate_bytes = gate.numel() * 4 if gate is not None else 0
        e2e = {"value": w.B * w.T * steps_e2e * world / dt, "unit": "tokens/s",
               "h2d_bytes_per_step": (qh.numel() + kh.numel() + vh.numel()) * es + gate_bytes,
               "d2h_bytes_per_step": oh.numel() * es, "steps": steps_e2e}
        del qh, kh, vh, oh

    decode = None if args.no_decode else _bench_decode(kg, peaks, args)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        keep = min(w.B * w.H, 4)
        sub = w.scaled(B=1, H=keep)
        BH = w.B * w.H
        qh = _host_f64(q.reshape(BH, w.T, w.d)[:keep]).reshape(1, keep, w.T, w.d)
        kh = _host_f64(k.reshape(BH, w.T, w.d)[:keep]).reshape(1, keep, w.T, w.d)
        vh = _host_f64(v.reshape(BH, w.T, w.dv)[:keep]).reshape(1, keep, w.T, w.dv)
        gh64 = None
        if gate is not None:
            gh64 = _host_f64(gate.reshape(BH, w.T)[:keep]).reshape(1, keep, w.T)
        nrows, dt, threads = _oracle_sample(sub, qh, kh, vh, args.cpu_seconds,
                                            np.random.default_rng(1), fm, gh64)
        # each row is one head; a token of the workload has H heads
        tps = (nrows / w.H) / dt
        cpu = {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{nrows} output rows from heads 0..{keep - 1}, positions uniform in "
                         f"[0,T), direct O(T^2) fp64 definition"
                         f"{' (gated)' if gh64 is not None else ''}, {dt:.1f} s; tokens = rows / H"}
        cpu.update(_cpu_extras(sub, qh, kh, vh, args.cpu_seconds, fm, gh64))

    if rank == 0:
        line = {
            "metric": _metric(), "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": _dtype_name(w), "data": "synthetic",
            "config": dict(_config(w, fm), algorithm=args.algo),
            "path": {0: "none", 1: "simt", 2: "tcgen05"}.get(path, str(path)),
            "roofline": roofline, "whole_call": whole, "cpu_baseline": cpu, "e2e": e2e,
            "decode": decode, "clocks": clk.summary(), "gpu_launches": launches,
            "stages": {k_: {"launches": n_, "total_ms": t_} for k_, (n_, t_) in stages.items()},
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def _bench_decode(kg, peaks, args):
    w = workloads.DECODE
    S, z = workloads.make_decode_state_fill(w, device="cuda")
    q, k, v = workloads.make_decode_inputs(w, device="cuda")
    o = torch.empty(w.B, w.H, w.dv, dtype=w.dtype, device="cuda")
    for _ in range(3):
        kg.kata_decode_step(S, z, q, k, v, out=o)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(5, args.steps)
    a.record(stream)
    for _ in range(steps):
        kg.kata_decode_step(S, z, q, k, v, out=o)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    BH, n = w.B * w.H, w.n
    nbytes = BH * (2 * 4 * n * w.dv + 2 * 4 * n) + BH * (2 * w.d + 2 * w.dv) * 2
    gbs = nbytes / (ms / 1e3) / 1e9
    # the GatedKATA step: the same sweep with a per-head gate (4 more bytes per head)
    g = workloads.make_decode_gate(w, device="cuda")
    for _ in range(3):
        kg.kata_decode_step_gated(S, z, q, k, v, g, out=o)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        kg.kata_decode_step_gated(S, z, q, k, v, g, out=o)
    b.record(stream)
    torch.cuda.synchronize()
    ms_g = a.elapsed_time(b) / steps
    gbs_g = (nbytes + 4 * BH) / (ms_g / 1e3) / 1e9
    return {"workload": "decode B=256 H=16 d=64 dv=64 fp32 state", "ms_per_step": ms,
            "tokens_per_s": w.B / (ms / 1e3),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "bytes_per_step": nbytes},
            "gated": {"ms_per_step": ms_g, "achieved_gbs": gbs_g,
                      "frac": gbs_g / peaks["hbm_gbs"]}}


def run_scan_ubench(args):
    """Chunk-scan micro-benchmark at the pages' small-batch linear-state shape
    (B=1, H=16, d=64, dv=64, C=128, orthant map, bf16 inputs, T from 2k to 64k):
    the forward with the one-pass chunk scan and with the two-level scan
    (KATA_CHUNK_SCAN), one JSON line per (T, scan); inputs resident, no flush."""
    from kernelized_causal_linear_gb300 import build
    build.build()
    import kernelized_causal_linear_gb300 as kg
    fm = FeatureMap("orthant")
    stream = torch.cuda.current_stream()
    for T in (2048, 8192, 32768, 65536):
        w = workloads.WORKLOADS["long_ctx_bf16"].scaled(B=1, H=16, T=T, d=64, dv=64, C=128)
        q, k, v = workloads.make_qkv(w, device="cuda")
        out = torch.empty(w.B, w.H, w.T, w.dv, dtype=w.dtype, device="cuda")
        for mode in ("sequential", "blocked"):
            os.environ["KATA_CHUNK_SCAN"] = mode
            for _ in range(max(3, args.warmup)):
                kg.kata_fwd_chunked_map(q, k, v, w.C, fm.code, 1, fm.eps, out=out)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            kg.kata_trace_begin()
            a.record(stream)
            for _ in range(args.steps):
                kg.kata_fwd_chunked_map(q, k, v, w.C, fm.code, 1, fm.eps, out=out)
            b.record(stream)
            torch.cuda.synchronize()
            stages = kg.kata_trace_end()
            ms = a.elapsed_time(b) / args.steps
            scan = {k_: t_ / n_ for k_, (n_, t_) in stages.items() if "scan" in k_}
            print(json.dumps({"ubench": "chunk_scan", "T": T, "scan": mode, "ms_per_call": ms,
                              "Mtok_s": w.B * w.T / ms / 1e3, "scan_ms": scan,
                              "config": _config(w, fm)}), flush=True)
        os.environ.pop("KATA_CHUNK_SCAN", None)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--map", default="full", choices=["full", "M", "Sigma", "orthant"],
                    help="feature map: the full rank-one map or a reduced PSD family")
    ap.add_argument("--g", type=int, default=1, help="blocks of the reduced map (1, 2 or 4)")
    ap.add_argument("--algo", default="chunked",
                    choices=["chunked", "quadratic", "gated", "gated_quadratic"],
                    help="chunked O(T) form (the default), the quadratic flash-style form, "
                         "GatedKATA chunked (tensor cores for bf16, else CUDA cores) or "
                         "GatedKATA quadratic (tensor cores); the gated forms draw seeded gates")
    ap.add_argument("--shape", default=None, metavar="B,H,T",
                    help="the workload's recipe at another batch, head count and length "
                         "(for profiles of other shapes; the bench line uses the named sizes)")
    ap.add_argument("--head-dims", default=None, metavar="d,dv",
                    help="the workload's recipe at another head size (d in 16, 32, 64; dv in "
                         "16, 32, 64, 128), for timings of the other shapes the library takes")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--ubench", choices=["scan"], default=None,
                    help="micro-benchmark instead of the bench line: 'scan' compares the "
                         "one-pass and the two-level chunk scan at small-batch shapes")
    args = ap.parse_args(argv)
    if args.shape is not None:
        try:
            b_, h_, t_ = (int(x) for x in args.shape.split(","))
        except ValueError:
            ap.error("--shape takes B,H,T")
        args.shape = (b_, h_, t_)
    if args.head_dims is not None:
        try:
            d_, dv_ = (int(x) for x in args.head_dims.split(","))
        except ValueError:
            ap.error("--head-dims takes d,dv")
        args.head_dims = (d_, dv_)
    if args.ubench == "scan":
        return run_scan_ubench(args)
    if args.map == "full" and args.g != 1:
        ap.error("--map full takes --g 1")
    if args.algo != "chunked" and args.map != "full":
        ap.error(f"--algo {args.algo} runs the full map")
    if args.warmup < 3:
        sys.stderr.write("warning: fewer than 3 warm-up steps\n")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
