"""Benchmark of the draft -> verify -> accept round on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mistral|qwen|llama|stagger|tiny]
                    [--impl ours|reference] [--schedule staggered|lockstep]

One step = one decode round of the whole hot path on one batch of synthetic
inputs: k draft steps over the packed cache (every layer), the full KV of every
layer streamed host->device in chunks (overlapped with drafting), verify
attention, accept, and the commit of the accepted tokens to the full-KV store
and the draft cache (with packing of full tail groups).  Per-round inputs
(queries, the new tokens' K/V, logits) are device-resident for ``value`` and
copied from pinned host memory inside the timed region for ``e2e``.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead (the reference arm).
Under torchrun each rank runs an independent replica (no data-path
collective); value = total over ranks, timed as max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified tokens/s/layer"
PCIE_GEN5_GBS = 64.0
L2_BYTES = 129 * 2 ** 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d.get("hbm_gbs", 6800.0), "bf16_tflops": d.get("bf16_tflops", 1900.0),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", 1700.0),
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
            "source": "fallback"}


# ---------------------------------------------------------------- clocks sampler
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, interval_ms=50):
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def wait_ready(self, n=3, timeout=10.0):
        """Block until the sampler has printed ``n`` samples: its start-up (driver
        initialisation) stalls the GPU's host interface for tens of ms and must
        not land inside the timed region."""
        t_end = time.time() + timeout
        while self.proc is not None and len(self.lines) < n and time.time() < t_end:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0=None, t1=None):
        """Stop sampling; summarise the samples that arrived in [t0, t1] (wall time)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if t0 is not None and not (t0 - 0.25 <= ts <= t1 + 0.25):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- inputs
def make_round_inputs(w, rnd, group, device, layers):
    import numpy as np
    import torch

    import synth
    from verify_compressed_kv_gb300.runtime import RoundInputs

    def t(a, dt=None):
        a = np.ascontiguousarray(a)
        v = {np.dtype(np.uint16): np.int16}.get(a.dtype, a.dtype)
        return torch.from_numpy(a.view(v))

    qd = np.stack([np.stack([synth.draft_q(w, rnd, i, l, group) for i in range(w.k)]) for l in range(layers)])
    kc = [[synth.draft_kv_cur(w, rnd, i, l, group) for i in range(w.k)] for l in range(layers)]
    kvc = np.stack([np.stack([np.stack([kc[l][i][j] for i in range(w.k)]) for l in range(layers)]) for j in range(2)])
    qv = np.stack([synth.verify_q(w, rnd, l, group) for l in range(layers)])
    kn = [synth.kv_new(w, rnd, l, group) for l in range(layers)]
    kvn = np.stack([np.stack([kn[l][j] for l in range(layers)]) for j in range(2)])
    logits, drafts, _ = synth.logits_and_drafts(w, rnd, group)
    host = RoundInputs(t(qd), t(kvc), t(qv), t(kvn), t(logits), t(drafts))
    return host


def round_drafts(w, host_inputs, n_rounds, group):
    """Draft tokens int32 [B, k] of rounds 0 .. n_rounds - 1 of one group, over the
    logits of input slot r % n_inp: the slot's row argmaxes (lowest index) below the
    round's accepted length L, drawn from the workload's distribution
    (synth.accept_lengths(w, r)), and a mismatch from L on.  A few input slots then
    still give the distribution's mean accepted length; the accept kernel finds n = L
    from the logits."""
    import numpy as np
    import torch

    import synth
    amax = [hi.logits.numpy().argmax(-1).astype(np.int64) for hi in host_inputs]     # [B, k+1] per slot
    out = []
    for r in range(n_rounds):
        A = amax[r % len(amax)]
        L = synth.accept_lengths(w, r, group)
        d = ((A[:, :w.k] + 1) % w.V).astype(np.int32)          # mismatches everywhere ...
        for b in range(w.B):
            d[b, :int(L[b])] = A[b, :int(L[b])]                # ... except below L
        out.append(torch.from_numpy(d))
    return out


def with_drafts(inp, drafts):
    import dataclasses
    return dataclasses.replace(inp, drafts=drafts)


def to_device(inp, device, pinned=False):
    from verify_compressed_kv_gb300.runtime import RoundInputs
    f = (lambda x: x.pin_memory()) if pinned else (lambda x: x.to(device))
    return RoundInputs(*[f(getattr(inp, n)) for n in ("q_draft", "kv_cur", "q_verify", "kv_new", "logits", "drafts")])


ALL_FIELDS = ("q_draft", "kv_cur", "q_verify", "kv_new", "logits", "drafts")
DRAFT_FIELDS = ("q_draft", "kv_cur", "drafts")                  # what a drafting round reads
VERIFY_FIELDS = ("q_verify", "kv_new", "logits", "drafts")      # what verify, accept and commit read


def copy_inputs(dst, src, stream, fields=ALL_FIELDS):
    import torch
    with torch.cuda.stream(stream):
        for n in fields:
            getattr(dst, n).copy_(getattr(src, n), non_blocking=True)


def input_bytes(inp, fields=ALL_FIELDS):
    return sum(getattr(inp, n).numel() * getattr(inp, n).element_size() for n in fields)


def build_group(w, layers, device, rounds_total, n_slots, group_index=0):
    import numpy as np
    import torch

    import synth
    from verify_compressed_kv_gb300.runtime import Group

    from verify_compressed_kv_gb300 import _lib as vc

    drop = w.keep_frac < 1.0
    g = Group(w.B, w.Hq, w.Hkv, w.d, w.k, w.bits, w.V, w.C, w.T, layers=layers,
              extra_tokens=(rounds_total + 2) * (w.k + 1), n_slots=n_slots, softmax_scale=1.0, device=device,
              packed_T0=w.T_keep if drop else None)
    for l in range(layers):
        K, V = synth.kv(w, layer=l, group=group_index, threads=16)
        Kd = torch.from_numpy(K.view(np.int16)).to(device)
        Vd = torch.from_numpy(V.view(np.int16)).to(device)
        if not drop:
            g.load_prefix(l, Kd, Vd)
        else:
            # token dropping (score -> select -> gather), then 4-bit packing of the kept tokens
            keep = w.T_keep
            qo = torch.from_numpy(synth.q_obs(w, group=group_index).view(np.int16)).to(device)
            score = torch.empty((w.B, w.Hkv, w.T), dtype=torch.float32, device=device)
            wsb = vc.vc_token_score_workspace_size(g.shape, w.T, 32)
            ws = torch.empty(wsb, dtype=torch.uint8, device=device)
            vc.vc_token_score(g.shape, w.T, 32, qo, Kd, score, ws, wsb)
            wsb2 = vc.vc_token_select_workspace_size(w.B, w.Hkv, w.T)
            ws2 = torch.empty(wsb2, dtype=torch.uint8, device=device)
            idx = torch.empty((w.B, w.Hkv, keep), dtype=torch.int32, device=device)
            vc.vc_token_select(w.B, w.Hkv, w.T, score, keep, 32, 7, idx, ws2, wsb2)
            Kk = torch.empty((w.B, w.Hkv, keep, w.d), dtype=torch.int16, device=device)
            Vk = torch.empty_like(Kk)
            vc.vc_gather_kv(g.shape, w.T, keep, idx, Kd, Vd, Kk, Vk)
            g.load_packed_only(l, Kk, Vk)
            g.write_store(l, Kd, Vd)
            del Kk, Vk, score, ws, ws2
        del Kd, Vd
    torch.cuda.synchronize()
    return g


# ---------------------------------------------------------------- our arm
def algorithmic_draft_bytes(w, P):
    """Bytes one draft call must move: packed K/V codes + metadata of P tokens per
    (request, KV head), plus q in and o out (the bf16 tail is < 1%: ignored)."""
    per_tok = 2 * w.d * w.bits // 8 + 2 * (w.d // 32) * 4
    return w.B * w.Hkv * P * per_tok + 2 * w.B * w.Hq * w.d * 2


def bench_config(w, args, world):
    """The bench line's `config` (the same dict in both arms): the workload, its
    schedule, and how the timed region stays clear of L2."""
    P = w.T_keep if w.name == "qwen" else w.T
    packed_mib = algorithmic_draft_bytes(w, P) * w.layers // 2 ** 20
    full_mib = 2 * w.B * w.Hkv * w.T * w.d * 2 * w.layers // 2 ** 20
    return {"workload": workload_name(w), "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "T": w.T, "k": w.k,
            "bits": w.bits, "layers": w.layers, "groups": w.groups, "V": w.V, "chunk": w.C,
            "schedule": "single" if w.groups == 1 else args.schedule,
            "l2": "inputs larger than L2 (packed cache %d MiB, full KV %d MiB per round)" % (packed_mib, full_mib),
            "parallelism": "replicas" if world > 1 else "single"}


def source_hash(path):
    """Hash of a kernel source's code: comments and whitespace removed, so edits to
    the comments keep a capture valid and any change to the code does not."""
    import re
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256("".join(text.split()).encode()).hexdigest()[:16]


def ncu_traffic(kernel_file, workload, alg_bytes):
    """DRAM bytes of one draft launch moving `alg_bytes` algorithmic bytes, from
    the committed ncu summary if it was taken on the current source of the
    kernel (else None).  The capture's launch (one layer of the workload at
    its prefix length) moves the summary's algorithmic bytes; the launches a
    bench times carry the tokens the rounds appended, and the DRAM bytes are
    scaled by the ratio of algorithmic bytes (the kernel reads every packed
    byte once, so its traffic grows in proportion)."""
    prof = os.path.join(ROOT, "profiles", f"draft_attn_{workload}.md")
    if not os.path.exists(prof):
        return None
    kv = {}
    for line in open(prof):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_sha256_16") != source_hash(kernel_file):
        return None
    try:
        return float(kv["dram_bytes_per_launch"]) * alg_bytes / float(kv["algorithmic_bytes_per_launch"])
    except (KeyError, ValueError, ZeroDivisionError):
        return None


def measure_link_gbs(device, stream, mib=512, reps=4):
    """The link's own peak: best pinned host->device copy of `mib` MiB (the
    roofline of the H2D stream), measured on this machine at this moment."""
    import torch
    h = torch.empty(mib * 2 ** 20, dtype=torch.uint8, pin_memory=True)
    h.fill_(1)
    d = torch.empty_like(h, device=device)
    best = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            d.copy_(h, non_blocking=True)
            e1.record(stream)
        e1.synchronize()
        best = max(best, h.numel() / e0.elapsed_time(e1) / 1e6)
    del h, d
    return best


def time_kernel(fn, stream, reps=20, warm=3):
    """Average CUDA-event time (ms) of fn() on `stream`."""
    import torch
    for _ in range(warm):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps


def time_token_drop(w, shape, Kd, Vd, device, cs):
    """Score, select and gather of the token-dropping compressor on layer 0,
    each timed alone against its roofline."""
    import numpy as np
    import torch

    import synth
    from verify_compressed_kv_gb300 import _lib as vc
    peaks = load_peaks()
    keep = w.T_keep
    qo = torch.from_numpy(synth.q_obs(w).view(np.int16)).to(device)
    score = torch.empty((w.B, w.Hkv, w.T), dtype=torch.float32, device=device)
    wsb = vc.vc_token_score_workspace_size(shape, w.T, 32)
    ws = torch.empty(wsb, dtype=torch.uint8, device=device)
    t_score = time_kernel(lambda: vc.vc_token_score(shape, w.T, 32, qo, Kd, score, ws, wsb, cs), cs, reps=5)
    flops = 4.0 * w.B * w.Hq * 32 * w.T * w.d            # QK in both passes, 2 flops per multiply-add
    wsb2 = vc.vc_token_select_workspace_size(w.B, w.Hkv, w.T)
    ws2 = torch.empty(wsb2, dtype=torch.uint8, device=device)
    idx = torch.empty((w.B, w.Hkv, keep), dtype=torch.int32, device=device)
    t_sel = time_kernel(lambda: vc.vc_token_select(w.B, w.Hkv, w.T, score, keep, 32, 7, idx, ws2, wsb2, cs), cs, reps=5)
    Ko = torch.empty((w.B, w.Hkv, keep, w.d), dtype=torch.int16, device=device)
    Vo = torch.empty_like(Ko)
    t_gat = time_kernel(lambda: vc.vc_gather_kv(shape, w.T, keep, idx, Kd, Vd, Ko, Vo, cs), cs, reps=10)
    gat_bytes = 2 * 2 * w.B * w.Hkv * keep * w.d * 2
    # K is read once per pass (2 bytes a channel), the scores written once: at
    # 32*G flops per byte the score sits below the bf16 ridge, so HBM bounds it
    score_bytes = 2 * w.B * w.Hkv * w.T * w.d * 2 + w.B * w.Hkv * w.T * 4
    return {"a3_token_score": dict(intensity_row(t_score, flops, score_bytes, peaks), engine="tcgen05 bf16"),
            "a4_token_select": {"ms": t_sel, "bound": "latency (6 passes over the pooled scores)"},
            "a4_gather": {"ms": t_gat, "gbs": gat_bytes / (t_gat / 1e3) / 1e9, "bound": "hbm",
                          "frac": gat_bytes / (t_gat / 1e3) / 1e9 / peaks["hbm_gbs"]}}


def intensity_row(t_ms, flops, nbytes, peaks):
    """A contraction kernel against its roofline: HBM when its arithmetic
    intensity (flops per byte it must move) is below the bf16 ridge point
    (tensor peak / HBM peak), else the tensor peak."""
    tflops = flops / (t_ms / 1e3) / 1e12
    gbs = nbytes / (t_ms / 1e3) / 1e9
    intensity = flops / nbytes
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    hbm = intensity < ridge
    return {"ms": t_ms, "tflops": tflops, "gbs": gbs, "flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
            "bound": "hbm" if hbm else "tensor (bf16)",
            "frac": gbs / peaks["hbm_gbs"] if hbm else tflops / peaks["bf16_tflops"]}


def verify_row(t_ms, flops, chunk_bytes, peaks, link_gbs):
    """The verify chunk kernel against its roofline (intensity_row: the chunk's
    bytes), plus the time the link takes to deliver that chunk."""
    return dict(intensity_row(t_ms, flops, chunk_bytes, peaks), chunk_transfer_ms=chunk_bytes / (link_gbs * 1e6))


def time_full_kv_resident(g, q1, kv1, out1, layers, cs, n_dec=3):
    """Context line: greedy decoding with every layer's full KV resident in HBM
    (its chunks copied once into the layer's ring), one token per request per
    step through the same verify kernels (k = 0): what a GPU that holds the KV
    does without the host link."""
    import torch

    from verify_compressed_kv_gb300 import _lib as vc
    n_chunks = g.chunks()
    if g.n_slots < n_chunks:
        return {"value": None, "why": f"ring of {g.n_slots} slots per layer < {n_chunks} chunks"}
    sh0 = vc.shape(g.B, g.Hq, g.Hkv, g.d, k=0, bits=g.bits, softmax_scale=g.shape.softmax_scale)
    parts0 = vc.vc_verify_attn_parts(sh0, g.C)
    wsb = vc.vc_verify_attn_workspace_size(sh0, parts0)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=g.device)
    n = n_chunks * g.chunk_elems
    for l in range(layers):
        g.ring[l][:n].copy_(g.host_kv[l][:n])            # once, outside the timed steps
    torch.cuda.synchronize()

    def step():
        for l in range(layers):
            for c in range(n_chunks):
                vc.vc_verify_attn_chunk(sh0, q1[l], g.ring[l][c * g.chunk_elems:], g.C, c * g.C, g.prefix_len[l],
                                        parts0, c == 0, ws, wsb, cs)
            vc.vc_verify_attn_finish(sh0, q1[l], kv1[0, l], kv1[1, l], parts0, True, out1, ws, wsb, cs)

    ms = time_kernel(step, cs, reps=n_dec, warm=2)
    kv_bytes = layers * 2 * g.B * g.Hkv * g.max_prefix * g.d * 2
    return {"value": g.B * layers / (ms / 1e3), "unit": "tokens/s/layer", "ms_per_step": ms,
            "kv_gbs": kv_bytes / (ms / 1e3) / 1e9,
            "what": "greedy decoding with the full KV resident in HBM (no link), same kernels, k = 0"}


def time_prefill_rows(w, shape, device, cs):
    """The prefill rows of layer 0, each timed alone: quantise + pack of the full
    prefix and, for the token-dropping compressor, score / select / gather."""
    import numpy as np
    import torch

    import synth
    from verify_compressed_kv_gb300 import _lib as vc
    peaks = load_peaks()
    K0, V0 = synth.kv(w, layer=0, group=0, threads=16)
    K0d = torch.from_numpy(K0.view(np.int16)).to(device)
    V0d = torch.from_numpy(V0.view(np.int16)).to(device)
    sb = vc.vc_quant_packed_bytes(shape, w.T)             # scratch packed arrays for the timing
    scratch = [torch.empty(n, dtype=torch.uint8, device=device) for n in sb]
    pack_ms = time_kernel(lambda: vc.vc_quant_kv_pack(shape, w.T, w.T, K0d, V0d, *scratch, cs), cs, reps=5)
    pack_bytes = 2 * w.B * w.Hkv * w.T * w.d * 2 + sum(sb)
    rows = {"a1_pack": {"ms": pack_ms, "gbs": pack_bytes / (pack_ms / 1e3) / 1e9, "bound": "hbm",
                        "frac": pack_bytes / (pack_ms / 1e3) / 1e9 / peaks["hbm_gbs"]}}
    if w.keep_frac < 1.0:
        rows.update(time_token_drop(w, shape, K0d, V0d, device, cs))
    del K0d, V0d, scratch
    torch.cuda.synchronize()
    return rows


def run_kernel(args, local_rank):
    """--kernel draft|verify|accept: one kernel alone on one layer of the
    workload, `--calls` back-to-back launches timed with CUDA events (a small
    device footprint and few launches, e.g. for ncu captures of that kernel).
    draft: vc_draft_attn over the layer's packed prefix (Qwen: the kept
    tokens), the current token only in the tail, calls chained as in a round.
    verify: vc_verify_attn_chunk on one resident chunk of the exact K/V.
    accept: vc_accept on the round's logits and drafts."""
    import numpy as np
    import torch

    import synth
    from verify_compressed_kv_gb300 import _lib as vc
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    w = workload_of(args)
    peaks = load_peaks()
    cs = torch.cuda.Stream(device)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device)
    calls = max(1, args.calls)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    if args.kernel == "draft":
        T = w.T_keep if w.keep_frac < 1.0 else w.T
        shape = vc.shape(w.B, w.Hq, w.Hkv, w.d, w.k, w.bits, 1.0 / math.sqrt(w.d))
        K, V = synth.kv(w, layer=0, group=0, T=T, threads=16)
        packed = [torch.zeros(n, dtype=torch.uint8, device=device) for n in vc.vc_quant_packed_bytes(shape, T)]
        vc.vc_quant_kv_pack(shape, T, T, dev(K), dev(V), *packed, cs)
        del K, V
        tail_cap = 32 + w.k + 1
        tk = torch.zeros((w.B, w.Hkv, tail_cap, w.d), dtype=torch.int16, device=device)
        tv = torch.zeros_like(tk)
        plen = torch.full((w.B,), T, dtype=torch.int32, device=device)
        tlen = torch.zeros(w.B, dtype=torch.int32, device=device)
        q = dev(synth.draft_q(w, 0, 0))
        kcur, vcur = (dev(x) for x in synth.draft_kv_cur(w, 0, 0))
        out = torch.empty((w.B, w.Hq, w.d), dtype=torch.int16, device=device)
        wsb = vc.vc_draft_attn_workspace_size(shape, T)
        ws = torch.zeros(wsb, dtype=torch.uint8, device=device)

        def call(i):
            vc.vc_draft_attn(shape, q, kcur, vcur, *packed, plen, T, T, tk, tv, tlen, tail_cap, 0, out, ws, wsb, cs,
                             flags=vc.VC_DRAFT_CHAINED if i > 0 else 0)
        nbytes = algorithmic_draft_bytes(w, T)
        status = vc.vc_draft_attn_device_status
    elif args.kernel == "verify":
        C = w.C
        shape = vc.shape(w.B, w.Hq, w.Hkv, w.d, w.k, w.bits, 1.0 / math.sqrt(w.d))
        parts = vc.vc_verify_attn_parts(shape, C)
        wsb = vc.vc_verify_attn_workspace_size(shape, parts)
        ws = torch.zeros(wsb, dtype=torch.uint8, device=device)
        K, V = synth.kv(w, layer=0, group=0, T=C, threads=16)
        slot = torch.stack([dev(K), dev(V)])
        del K, V
        q = dev(synth.verify_q(w, 0))
        plen = torch.full((w.B,), 4 * C, dtype=torch.int32, device=device)

        def call(i):
            vc.vc_verify_attn_chunk(shape, q, slot, C, 0, plen, parts, True, ws, wsb, cs)
        nbytes = 2 * w.B * w.Hkv * C * w.d * 2
        status = vc.vc_verify_attn_device_status
    else:
        logits, drafts, _ = synth.logits_and_drafts(w, 0)
        lg = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).to(device)
        dr = torch.from_numpy(np.ascontiguousarray(drafts, np.int32)).to(device)
        n_acc = torch.zeros(w.B, dtype=torch.int32, device=device)
        nxt = torch.zeros_like(n_acc)
        wsb = vc.vc_accept_workspace_size(w.B, w.k, w.V)
        ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=device)

        def call(i):
            vc.vc_accept(w.B, w.k, w.V, lg, dr, n_acc, nxt, None, ws, wsb, cs)
        nbytes = lg.numel() * 4
        status = lambda: 0
    torch.cuda.synchronize()
    for i in range(3):
        call(i)
    ev[0].record(cs)
    for i in range(calls):
        call(3 + i)
    ev[1].record(cs)
    ev[1].synchronize()
    ms = ev[0].elapsed_time(ev[1]) / calls
    st = status()
    if st != 0:
        raise RuntimeError(f"device status {st:#x}")
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"workload": workload_name(w), "mode": "kernel", "kernel": args.kernel, "calls": calls, "ms_per_call": ms,
            "bytes_per_call": nbytes, "gbs": gbs, "frac_of_measured_hbm": gbs / peaks["hbm_gbs"],
            "data": "synthetic"}


def run_rows(args, local_rank):
    """--rows-only: the prefill rows of one layer, without the decode loop (a small
    device footprint, e.g. for kernel captures)."""
    import torch

    from verify_compressed_kv_gb300 import _lib as vc
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    w = workload_of(args)
    shape = vc.shape(w.B, w.Hq, w.Hkv, w.d, w.k, w.bits, 1.0)
    cs = torch.cuda.Stream(device)
    rows = time_prefill_rows(w, shape, device, cs)
    return {"workload": workload_name(w), "mode": "rows-only", "data": "synthetic", "rows": rows}


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import synth

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    from verify_compressed_kv_gb300 import _lib as vc
    from verify_compressed_kv_gb300 import runtime as rt

    w = workload_of(args)
    layers = w.layers
    n_groups = w.groups
    # capacity (full-KV store, rings, draft cache) for every round the run makes: the
    # warm-up, the timed rounds and the e2e leg's rounds
    rounds_total = args.warmup + 2 * args.steps + 1
    n_inp = min(3, rounds_total)
    n_slots = args.slots or None
    cs = torch.cuda.Stream(device)
    xs = torch.cuda.Stream(device)
    groups = [build_group(w, layers, device, rounds_total, n_slots, gi) for gi in range(n_groups)]
    host_inputs = [[make_round_inputs(w, r, gi, device, layers) for r in range(n_inp)] for gi in range(n_groups)]
    dev_inputs = [[to_device(x, device) for x in hi] for hi in host_inputs]
    pin_inputs = [[to_device(x, device, pinned=True) for x in hi] for hi in host_inputs]
    # device buffers the e2e leg copies into every round
    e2e_bufs = [to_device(hi[0], device) for hi in host_inputs]
    # per-round draft tokens (accepted lengths drawn per round, see round_drafts)
    n_draft_rounds = args.warmup + 2 * args.steps + 8
    host_drafts = [round_drafts(w, host_inputs[gi], n_draft_rounds, gi) for gi in range(n_groups)]
    dev_drafts = [[x.to(device) for x in hd] for hd in host_drafts]
    pin_drafts = [[x.pin_memory() for x in hd] for hd in host_drafts]
    torch.cuda.synchronize()

    link_best = measure_link_gbs(device, xs)
    measured_link = link_best if args.link_peak_gbs <= 0 else args.link_peak_gbs

    # ---- prefill rows timed once (layer 0)
    prefill_rows = time_prefill_rows(w, groups[0].shape, device, cs)

    state = {"round": 0}

    def one_round(e2e=False, timeline=None):
        r = state["round"]
        state["round"] += 1
        if n_groups == 1:
            g = groups[0]
            inp = with_drafts(dev_inputs[0][r % n_inp], dev_drafts[0][r])
            copy_in = None
            if e2e:
                # the round's inputs come over the link ahead of its full KV (on the copy
                # stream); only the drafting waits for them
                src = with_drafts(pin_inputs[0][r % n_inp], pin_drafts[0][r])
                copy_in = lambda st, src=src: copy_inputs(e2e_bufs[0], src, st)
                inp = e2e_bufs[0]
            tl = rt.round_single(g, inp, cs, xs, timeline, copy_in=copy_in)
            return tl, [g]
        if args.schedule == "lockstep":
            # every group drafts cycle r, then every group verifies it
            inps = [with_drafts(dev_inputs[gi][r % n_inp], dev_drafts[gi][r]) for gi in range(2)]
            if e2e:
                for gi in range(2):
                    copy_inputs(e2e_bufs[gi], with_drafts(pin_inputs[gi][r % n_inp], pin_drafts[gi][r]), cs)
                inps = e2e_bufs
            tl = rt.round_lockstep(groups, inps, cs, xs, timeline)
            return tl, list(groups)
        # staggered: round r, group r % 2 drafts its cycle r // 2 while the other
        # group verifies its cycle (r - 1) // 2; round 0 is the prologue (draft only)
        ix, iy = r % 2, (r + 1) % 2
        X, Y = groups[ix], groups[iy]
        dc, vcyc = r // 2, (r - 1) // 2
        inp_x = with_drafts(dev_inputs[ix][dc % n_inp], dev_drafts[ix][dc])
        if r == 0:
            tl = rt.Timeline()
            tl.mark("start", cs)
            for i in range(X.k):
                for l in range(X.L):
                    X.draft_step(inp_x, l, i, cs, chained=i + l > 0)
            tl.mark("end", cs)
            return tl, []
        inp_y = with_drafts(dev_inputs[iy][vcyc % n_inp], dev_drafts[iy][vcyc])
        copy_in = None
        if e2e:
            # each group copies what its role in this round reads, ahead of the full KV
            sx = with_drafts(pin_inputs[ix][dc % n_inp], pin_drafts[ix][dc])
            sy = with_drafts(pin_inputs[iy][vcyc % n_inp], pin_drafts[iy][vcyc])

            def copy_in(st, sx=sx, sy=sy, ix=ix, iy=iy):
                copy_inputs(e2e_bufs[ix], sx, st, DRAFT_FIELDS)
                copy_inputs(e2e_bufs[iy], sy, st, VERIFY_FIELDS)
            inp_x, inp_y = e2e_bufs[ix], e2e_bufs[iy]
        tl = rt.round_staggered(X, Y, inp_x, inp_y, cs, xs, timeline, copy_in=copy_in)
        return tl, [Y]

    def finish(tl, done):
        tl.ev["end"].synchronize()
        return sum(g.after_round() for g in done)

    # ---- warm-up (the clock sampler starts first: its start-up must not fall
    # inside the timed region)
    clocks = Clocks(local_rank, args.clock_ms)
    clocks.start()
    clocks.wait_ready()
    time.sleep(0.5)
    for _ in range(args.warmup):
        tl, done = one_round()
        finish(tl, done)
    torch.cuda.synchronize()

    # ---- timed region (device-resident per-round inputs)
    dist_barrier(world)
    torch.cuda.synchronize()
    launches0 = sum(g.launches for g in groups)
    wall0 = time.time()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(cs)
    tokens = 0
    tls = []
    h2d_bytes = 0
    for _ in range(args.steps):
        h2d_bytes += sum(g.h2d_bytes() for g in (groups if (n_groups == 1 or args.schedule == "lockstep")
                                                 else [groups[1] if state["round"] % 2 == 0 else groups[0]]))
        tl, done = one_round()
        tokens += finish(tl, done)
        tls.append(tl)
    t_end.record(cs)
    torch.cuda.synchronize()
    wall1 = time.time()
    clk = clocks.stop(wall0, wall1)
    dist_barrier(world)
    launches = sum(g.launches for g in groups) - launches0
    total_ms = t_start.elapsed_time(t_end)
    layer_tokens = tokens * layers
    value_local = layer_tokens / (total_ms / 1e3)

    # ---- e2e: the same rounds right after the device-resident ones (same state of the
    # group and its rings), inputs copied from pinned host memory every round, result read back
    dist_barrier(world)
    torch.cuda.synchronize()
    e2e_tokens = 0
    e2e_tls = []
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(cs)
    for _ in range(args.steps):
        tl, done = one_round(e2e=True)
        e2e_tokens += finish(tl, done)
        e2e_tls.append(tl)
    s1.record(cs)
    torch.cuda.synchronize()
    e2e_ms = s0.elapsed_time(s1)
    e2e_local = e2e_tokens * layers / (e2e_ms / 1e3)
    if n_groups == 1 or args.schedule == "lockstep":
        per_round_in = input_bytes(pin_inputs[0][0]) * n_groups
    else:                                       # staggered: one group's draft inputs, the other's verify inputs
        per_round_in = input_bytes(pin_inputs[0][0], DRAFT_FIELDS) + input_bytes(pin_inputs[0][0], VERIFY_FIELDS)
    per_round_out = 4 * w.B

    # per-round breakdown from the timelines
    def med(xs_):
        return statistics.median(xs_) if xs_ else None
    draft_span = [tl.ms("draft_start", "draft_end") for tl in tls]
    copy_span = [tl.ms("copy_start", "copy_end") for tl in tls]
    overlap = []
    for tl in tls:
        a0, a1 = tl.ms("start", "draft_start"), tl.ms("start", "draft_end")
        b0, b1 = tl.ms("start", "copy_start"), tl.ms("start", "copy_end")
        inter = max(0.0, min(a1, b1) - max(a0, b0))
        overlap.append(inter / max(1e-9, b1 - b0))
    round_ms = [tl.ms("start", "end") for tl in tls]
    commit_span = [tl.ms("commit_start", "commit_end") for tl in tls if "commit_start" in tl.ev]

    # ---- the draft call alone, timed on its stream (CUDA events, L2 > inputs):
    # back-to-back calls chained as in a round (each may start while the
    # previous one finishes), and the same calls each waiting for the previous
    g = groups[0]
    inp = dev_inputs[0][0]
    n_draft = 20

    def draft_calls_ms(chained):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for i in range(3):
            g.draft_step(inp, 0, 0, cs, chained=chained and i > 0)
        ev[0].record(cs)
        for i in range(n_draft):
            g.draft_step(inp, 0, 0, cs, chained=chained)
        ev[1].record(cs)
        ev[1].synchronize()
        return ev[0].elapsed_time(ev[1]) / n_draft
    draft_unchained_ms = draft_calls_ms(False)
    draft_call_ms = draft_calls_ms(True)
    P = int(g.packed_len[0].max().item())
    alg_bytes = algorithmic_draft_bytes(w, P)
    peaks = load_peaks()
    achieved_gbs = alg_bytes / (draft_call_ms / 1e3) / 1e9
    # inside the timed rounds: average draft call = draft span / (k * layers)
    draft_in_round_ms = med(draft_span) / (w.k * layers)

    # ---- the other rows of the path, each timed alone against its roofline
    g.ring[0][:g.chunk_elems].copy_(g.host_kv[0][:g.chunk_elems])     # one resident chunk
    torch.cuda.synchronize()
    t_ver = time_kernel(lambda: vc.vc_verify_attn_chunk(g.shape, inp.q_verify[0], g.ring[0], g.C, 0, g.prefix_len[0],
                                                        g.parts, True, g.ws_verify, g.ws_verify_bytes, cs), cs)
    ver_flops = 4.0 * w.B * w.Hq * (w.k + 1) * w.C * w.d               # QK and PV of (k+1)*Hq rows x C tokens
    t_acc = time_kernel(lambda: g.accept(inp, cs), cs)
    acc_bytes = w.B * (w.k + 1) * w.V * 4
    rows = {
        "a5_draft": {"ms": draft_call_ms, "gbs": achieved_gbs, "bound": "hbm", "frac": achieved_gbs / peaks["hbm_gbs"]},
        "a7_verify_chunk": verify_row(t_ver, ver_flops, g.chunk_elems * 2, peaks, measured_link),
        "a8_accept": {"ms": t_acc, "gbs": acc_bytes / (t_acc / 1e3) / 1e9, "bound": "hbm",
                      "frac": acc_bytes / (t_acc / 1e3) / 1e9 / peaks["hbm_gbs"]},
    }
    rows.update(prefill_rows)

    # ---- context: plain full-KV decoding (one token per request per step), the
    # full KV of every layer streamed from pinned host memory each step as in the
    # pages' long-context scenario, through the same streamed verify kernel (k = 0)
    g = groups[0]
    inp0 = dev_inputs[0][0]
    q1 = inp0.q_verify[:, :, :1].contiguous()
    kv1 = inp0.kv_new[:, :, :, :1].contiguous()
    out1 = torch.empty((w.B, 1, w.Hq, w.d), dtype=torch.int16, device=device)
    n_dec = 3
    for _ in range(2):
        for l in range(layers):
            g.decode_full_kv(q1[l], kv1[:, l], out1, l, cs, xs)
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    d0.record(cs)
    for _ in range(n_dec):
        for l in range(layers):
            g.decode_full_kv(q1[l], kv1[:, l], out1, l, cs, xs)
    ex = torch.cuda.Event()
    ex.record(xs)
    cs.wait_event(ex)
    d1.record(cs)
    d1.synchronize()
    dec_ms = d0.elapsed_time(d1) / n_dec
    full_kv = {"value": w.B * layers / (dec_ms / 1e3), "unit": "tokens/s/layer", "ms_per_step": dec_ms,
               "what": "greedy decoding with the full KV streamed host->device every step (same kernels, k = 0)"}
    full_kv_resident = time_full_kv_resident(g, q1, kv1, out1, layers, cs)

    # ---- reduce over ranks (replicas): value = sum, time = max
    value, e2e_value, t_max = reduce_over_ranks(value_local, e2e_local, total_ms, world)

    draft_src = os.path.join(ROOT, "verify_compressed_kv_gb300", "csrc", "vc_draft_attn.cu")
    traffic = ncu_traffic(draft_src, args.workload, alg_bytes)
    link_peak = measured_link
    h2d_rate = (h2d_bytes / args.steps) / (med(copy_span) / 1e3) / 1e9 if copy_span else None
    out = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s/layer",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_max / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16/int%d->f32" % w.bits,
        "data": "synthetic (seeded; shapes and distributions of the workload; no weights)",
        "config": bench_config(w, args, world),
        "e2e": {"value": e2e_value, "unit": "tokens/s/layer", "h2d_bytes_per_step": per_round_in,
                "round_ms_median": med([tl.ms("start", "end") for tl in e2e_tls]),
                "copy_ms_median": med([tl.ms("copy_start", "copy_end") for tl in e2e_tls]),
                "tokens_per_round": e2e_tokens / max(1, args.steps), "tokens_per_round_value": tokens / max(1, args.steps),
                "d2h_bytes_per_step": per_round_out},
        "gpu_launches": launches,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": "vc_draft_attn (stream-K split, bf16 tail and combine in one grid), "
                               "back-to-back chained calls alone on its stream",
                     "bytes_per_launch": alg_bytes, "ms_per_launch": draft_call_ms,
                     "ms_per_launch_unchained": draft_unchained_ms,
                     "ms_per_launch_in_round": draft_in_round_ms, "peak_source": peaks["source"]},
        "h2d": {"gbs": h2d_rate, "bytes_per_round": h2d_bytes / args.steps, "copy_ms": med(copy_span),
                "slots_per_layer": groups[0].n_slots,
                "frac_of_measured_link": (h2d_rate / link_peak) if h2d_rate else None,
                "measured_link_gbs": link_peak, "link_peak_source": "measured at start-up (best of 4 x 512 MiB)"
                if args.link_peak_gbs <= 0 else "given on the command line", "frac_of_pcie_gen5_64": (h2d_rate / PCIE_GEN5_GBS) if h2d_rate else None,
                "overlap_with_draft": med(overlap)},
        "round_ms": {"median": med(round_ms), "draft": med(draft_span), "copy": med(copy_span),
                     "commit": med(commit_span), "commit_max": max(commit_span) if commit_span else None,
                     "all": [round(x, 3) for x in round_ms],
                     "host_gap_total": round(total_ms - sum(round_ms), 3)},
        "rows": rows,
        "full_kv_decode": dict(full_kv, speedup_of_value=value_local / full_kv["value"]),
        "full_kv_resident": full_kv_resident if full_kv_resident.get("value") is None else
        dict(full_kv_resident, speedup_of_value=value_local / full_kv_resident["value"]),
        "clocks": clk,
    }
    for gg in groups:
        gg.close()
    if rank == 0 and world == 1 and not args.no_adaptive:
        why = adaptive_skip_reason(w)
        out["adaptive"] = {"skipped": why} if why else adaptive_compare(args, device, w, 4)
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.workload, w)
    return out


def workload_of(args):
    """The workload, with --bits / --k overriding its code width / draft length."""
    import synth
    ov = {}
    if args.bits:
        ov["bits"] = args.bits
    if getattr(args, "k", 0):
        ov["k"] = args.k
    return synth.get(args.workload, **ov)


def workload_name(w):
    names = {"tiny": "tiny 1x(Hq4,Hkv1,d64) T512 k4 int4",
             "mistral": "Mistral-24B-shaped layer: B8 Hq32 Hkv8 d128 T32768 k16 int2",
             "qwen": "Qwen-32B-shaped layer: B16 Hq40 Hkv8 d128 T65536 (keep 25%) k32 int4",
             "llama": "Llama-70B-shaped 8 layers: B4 Hq64 Hkv8 d128 T131072 k32 int2",
             "stagger": "staggered mix: 2x B32 Hq32 Hkv8 d128 T32768 k24 int2"}
    name = names.get(w.name, w.name)
    own = {"tiny": 4, "mistral": 2, "qwen": 4, "llama": 2, "stagger": 2}.get(w.name)
    if own is not None and w.bits != own:
        name = name.replace(f"int{own}", f"int{w.bits}")
    own_k = {"tiny": 4, "mistral": 16, "qwen": 32, "llama": 32, "stagger": 24}.get(w.name)
    if own_k is not None and w.k != own_k:
        name = name.replace(f" k{own_k} ", f" k{w.k} ")
    return name


# ---------------------------------------------------------------- CPU oracle leg
# One unit of oracle work = one (request, KV head) of one round of one layer:
# a draft step over the packed prefix (timed once, counted k times) and the
# verify pass of the k+1 rows over the full prefix.  Both are linear in the
# prefix length, so a unit is timed on the first T_SAMPLE tokens of its slice
# and scaled to the workload's length.  Worker processes (one BLAS thread
# each) build their units, report "ready", and time them when the parent
# sends "go" to all of them at once: the all-cores figure is measured with
# every core busy on the same work.
T_SAMPLE = 32768

ORACLE_WORKER = r"""
import json, sys, time
sys.path.insert(0, {root!r})
import numpy as np
import synth
from oracle import kivi, attention
w = synth.get({wl!r})
T = {T_s}
G = w.G
prep = []
for b, h in {units!r}:
    k_, v_ = synth.kv_slice(w, b, h, T=T)
    K = k_[None, None]
    V = v_[None, None]
    qh = list(range(h * G, (h + 1) * G))
    kc, vc_ = synth.draft_kv_cur(w, 0, 0)
    kn, vn = synth.kv_new(w, 0)
    prep.append(dict(K=K, V=V, packed=kivi.quant_pack(K, V, w.bits), q=synth.draft_q(w, 0, 0)[b:b + 1][:, qh],
                     kc=kc[b:b + 1][:, [h]], vc=vc_[b:b + 1][:, [h]], qv=synth.verify_q(w, 0)[b:b + 1][:, :, qh],
                     kn=kn[b:b + 1][:, :, [h]], vn=vn[b:b + 1][:, :, [h]]))
tail = np.zeros((1, 1, 32 + w.k + 1, w.d), np.uint16)
print("ready", flush=True)
while sys.stdin.readline().strip() == "go":
    t_start = time.time()
    res = []
    for u in prep:
        t0 = time.perf_counter()
        attention.draft_attention(u["q"], *u["packed"], [T], tail, tail, [0], w.bits, 1.0,
                                  k_cur=u["kc"], v_cur=u["vc"], step=0)
        t1 = time.perf_counter()
        attention.verify_attention(u["qv"], u["K"], u["V"], u["kn"], u["vn"], [T], 1.0)
        res.append((t1 - t0, time.perf_counter() - t1))
    print(json.dumps(dict(units=res, t_start=t_start, t_end=time.time())), flush=True)
"""


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


class OracleSampler:
    """Worker processes holding oracle units; run() times all of them together."""

    def __init__(self, workload, unit_lists, T_s):
        import tempfile
        env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
        self.procs, self.errs = [], []
        for units in unit_lists:
            code = ORACLE_WORKER.format(root=ROOT, wl=workload, T_s=T_s, units=[tuple(u) for u in units])
            err = tempfile.TemporaryFile(mode="w+")
            self.errs.append(err)
            self.procs.append(subprocess.Popen([sys.executable, "-c", code], stdin=subprocess.PIPE,
                                               stdout=subprocess.PIPE, stderr=err, text=True, env=env))
        for i, p in enumerate(self.procs):
            if p.stdout.readline().strip() != "ready":
                self._fail(i)

    def _fail(self, i):
        self.errs[i].seek(0)
        msg = self.errs[i].read()[-300:]
        self.close()
        raise RuntimeError("oracle worker failed: " + msg)

    def run(self):
        """Per-unit (draft step, verify) seconds of every worker, and the wall time of the slowest."""
        for p in self.procs:
            p.stdin.write("go\n")
            p.stdin.flush()
        res = []
        for i, p in enumerate(self.procs):
            line = p.stdout.readline()
            if not line:
                self._fail(i)
            res.append(json.loads(line))
        wall = max(r["t_end"] for r in res) - min(r["t_start"] for r in res)
        return [u for r in res for u in r["units"]], wall

    def close(self):
        for p in self.procs:
            try:
                p.stdin.close()
                p.wait(timeout=60)
            except Exception:
                p.kill()
        for e in self.errs:
            e.close()


def oracle_round_units(w):
    """The (request, KV head) units of one round of one layer, in a fixed order."""
    return [(b, h) for h in range(w.Hkv) for b in range(w.B)]


def oracle_value(w, units, workers, t_accept, tokens):
    """tokens/s/layer of the oracle running a whole round on `workers` cores,
    from unit times measured with that many cores busy.

    A round of one layer is B*Hkv units (k draft steps + one verify pass each,
    scaled from the sampled length to the workload's) spread over the workers,
    plus the accept step of the B requests (one core)."""
    T_d = w.T_keep if w.name == "qwen" else w.T          # drafting reads the kept tokens
    T_s = min(w.T, T_SAMPLE)
    per_unit = statistics.mean(w.k * td * (T_d / T_s) + tv * (w.T / T_s) for td, tv in units)
    n_units = w.B * w.Hkv
    round_layer = math.ceil(n_units / workers) * per_unit + t_accept
    return tokens / round_layer, per_unit


def oracle_accept(w):
    """Tokens of round 0 (accepted lengths + 1, summed over requests) and the accept step's time."""
    import synth
    from oracle import accept as oacc
    logits, drafts, _ = synth.logits_and_drafts(w, 0)
    t0 = time.perf_counter()
    n, _, _ = oacc.accept(logits, drafts)
    return int((n + 1).sum()), time.perf_counter() - t0


def cpu_baseline(workload, workload_obj=None):
    """The oracle, as it stands, on the machine's host cores: the same seeded units
    timed on 1 thread and on every core, scaled to the metric's unit."""
    import synth
    w = workload_obj or synth.get(workload)
    cores = len(os.sched_getaffinity(0))
    T_s = min(w.T, T_SAMPLE)
    t0 = time.time()
    order = oracle_round_units(w)
    try:
        tokens, t_acc = oracle_accept(w)
        one = OracleSampler(w.name, [order[:2]], T_s)
        u1, wall1 = one.run()
        one.close()
        n_par = min(cores, len(order))
        par = OracleSampler(w.name, [[order[i]] for i in range(n_par)], T_s)
        uc, wallc = par.run()
        par.close()
    except RuntimeError as e:
        return {"value": None, "unit": "tokens/s/layer", "cores": cores, "kind": "oracle", "sample": str(e)}
    v1, pu1 = oracle_value(w, u1, 1, t_acc, tokens)
    vc, puc = oracle_value(w, uc, n_par, t_acc, tokens)
    return {"value": vc, "unit": "tokens/s/layer", "cores": n_par, "kind": "oracle",
            "value_1thread": v1, "cpu_model": cpu_model(), "cores_available": cores,
            "sample": (f"round 0, one layer: (request, KV head) units, each a draft step (counted {w.k} times) and "
                       f"the {w.k + 1}-row verify pass, timed on the first {T_s} tokens of the slice and scaled to "
                       f"T={w.T_keep if w.name == 'qwen' else w.T} (draft) / T={w.T} (verify); 1 thread: 2 units "
                       f"in one process; all cores: {n_par} units, one per process, started together; round = "
                       f"{w.B * w.Hkv} units over the cores + accept of {w.B} requests ({tokens} tokens), x{w.layers} "
                       f"layer(s); numpy fp64, 1 BLAS thread per process"),
            "seconds": {"unit_1thread": pu1, "unit_all_cores": puc, "accept": t_acc,
                        "sample_wall_1thread": wall1, "sample_wall_all_cores": wallc},
            "wall_s": time.time() - t0}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step runs one all-cores sample of
    the workload (one unit per core, started together) and converts it to
    tokens/s/layer exactly as the default line's cpu_baseline does."""
    if rank != 0:
        return None
    import synth
    w = workload_of(args)
    cores = len(os.sched_getaffinity(0))
    T_s = min(w.T, T_SAMPLE)
    order = oracle_round_units(w)
    n_par = min(cores, len(order))
    t_all = time.time()
    tokens, t_acc = oracle_accept(w)
    one = OracleSampler(w.name, [order[:2]], T_s)
    u1, _ = one.run()
    one.close()
    v1, _ = oracle_value(w, u1, 1, t_acc, tokens)
    par = OracleSampler(w.name, [[order[i]] for i in range(n_par)], T_s)
    for _ in range(args.warmup):
        par.run()
    vals, walls = [], []
    for _ in range(args.steps):
        uc, wall = par.run()
        vals.append(oracle_value(w, uc, n_par, t_acc, tokens)[0])
        walls.append(wall)
    par.close()
    v = statistics.median(vals)
    cb = {"value": v, "unit": "tokens/s/layer", "cores": n_par, "kind": "oracle", "value_1thread": v1,
          "cpu_model": cpu_model(), "cores_available": cores,
          "sample": (f"per step: {n_par} (request, KV head) units of round 0, one per process, started together; "
                     f"each a draft step (counted {w.k} times) and the {w.k + 1}-row verify pass on the first "
                     f"{T_s} tokens, scaled to the workload's length; round = {w.B * w.Hkv} units over the cores "
                     f"+ accept; median over steps")}
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s/layer", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(walls) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic (seeded)",
            "config": bench_config(w, args, world),
            "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "tokens/s/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.time() - t_all}


# ---------------------------------------------------------------- distributed plumbing
ADAPTIVE_BLOCK = 10          # rounds per block; the fixed and the controller arm alternate blocks
STALL_FRAC = 0.8             # a round whose copy ran below this share of the measured link stalled


def adaptive_skip_reason(w):
    if w.groups != 1:
        return "two request groups (staggered): the controller plans one group's rounds"
    if w.keep_frac < 1.0:
        return "token dropping: the packed prefix is not the full prefix the controller's cost model assumes"
    return None


def adaptive_compare(args, device, w, n_blocks):
    """Fixed draft length (the workload's k) against a per-round draft length
    chosen by the controller from the previous rounds' measured spans, on one
    group whose buffers hold up to --k-max draft tokens.  Same process, same
    prefix and seeds, alternating blocks of ADAPTIVE_BLOCK rounds (n_blocks,
    even, fixed first)."""
    import dataclasses
    import statistics

    import torch

    from verify_compressed_kv_gb300 import runtime as rt
    from verify_compressed_kv_gb300.schedule import DraftLengthController

    k_max = max(args.k_max, w.k)
    choices = sorted({w.k, k_max} | {c for c in range(4, k_max + 1, 4)})
    rounds_total = args.warmup + n_blocks * ADAPTIVE_BLOCK + 4
    g = build_group(dataclasses.replace(w, k=k_max), w.layers, device, rounds_total, args.slots or None)
    n_inp = 3
    host_in = {k: [make_round_inputs(dataclasses.replace(w, k=k), r, 0, device, w.layers) for r in range(n_inp)]
               for k in choices}
    inputs = {k: [to_device(x, device) for x in host_in[k]] for k in choices}
    n_rounds = rounds_total + 8
    drafts = {k: [x.to(device) for x in round_drafts(dataclasses.replace(w, k=k), host_in[k], n_rounds, 0)]
              for k in choices}
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    ctl = DraftLengthController(k_max=k_max, k_min=choices[0], choices=tuple(choices))

    link_gbs = measure_link_gbs(device, xs)

    # verify compute per row: the chunk kernel alone on a resident slot, at the
    # smallest and the largest draft length (slope = cost of one more row)
    from verify_compressed_kv_gb300 import _lib as vc
    g.ring[0][:g.chunk_elems].copy_(g.host_kv[0][:g.chunk_elems])   # chunk 0 of layer 0 into slot 0
    torch.cuda.synchronize()

    def chunk_ms(k, reps=20):
        sh = g.shape_k(k)
        q = inputs[k][0].q_verify[0]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for i in range(reps + 3):
            if i == 3:
                e0.record(cs)
            vc.vc_verify_attn_chunk(sh, q, g.ring[0], g.C, 0, g.prefix_len[0], g.parts, True, g.ws_verify,
                                    g.ws_verify_bytes, cs)
        e1.record(cs)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps
    k_lo, k_hi = choices[0], choices[-1]
    # the chunk kernel timed at every candidate k: its cost steps with the launch
    # geometry (rows per KV head decide warps per CTA and CTAs per SM), so a slope
    # between two k would misjudge the rest
    chunk_of_k = {k: chunk_ms(k) for k in choices}
    row_chunk_ms = max(0.0, (chunk_of_k[k_hi] - chunk_of_k[k_lo]) / (k_hi - k_lo))
    rate = {"bytes_per_ms": link_gbs * 1e6}

    def one(k, r):
        h2d_bytes = g.h2d_bytes()
        pf_bytes = g.prefetch_bytes()
        tl = rt.round_single(g, with_drafts(inputs[k][r % n_inp], drafts[k][r % n_rounds]), cs, xs)
        tl.ev["end"].synchronize()
        toks = g.after_round()
        d_ms, r_ms = tl.ms("draft_start", "draft_end"), tl.ms("start", "end")
        v_end = tl.ms("start", "verify_end")
        t_tail = max(0.0, r_ms - v_end)
        # the transfer alone, at the best rate the prefetched copies have reached (they
        # never wait for a slot): the link's capacity, which an occasional stall of the
        # shared host link must not move (a stalled round would make every later plan
        # hide longer drafting behind a transfer that is not really that long)
        pf_ms = tl.ms("copy_start", "prefetch_end")
        if pf_ms > 0 and pf_bytes > 0:
            rate["bytes_per_ms"] = max(rate["bytes_per_ms"], pf_bytes / pf_ms)
        t_copy = h2d_bytes / rate["bytes_per_ms"]
        # verify compute of k + 1 rows over every chunk of every layer (calibrated slope),
        # and the measured table for every candidate k
        t_verify = (k + 1) * row_chunk_ms * g.chunks() * g.L
        ctl.observe(g.n_acc_host.numpy(), k, t_step=d_ms / k, t_copy=t_copy, t_tail=t_tail, t_verify=t_verify)
        ctl.t_verify = {kk: v * g.chunks() * g.L for kk, v in chunk_of_k.items()}
        c_ms = tl.ms("copy_start", "copy_end")
        return toks, r_ms, (h2d_bytes / c_ms / 1e6 if c_ms > 0 else None)

    for r in range(args.warmup):
        one(w.k, r)
    res = {"fixed": [0, 0.0], "adaptive": [0, 0.0]}
    per_round = {"fixed": [], "adaptive": []}            # (tokens, ms) of every round
    stalled = {"fixed": 0, "adaptive": 0}
    chosen = {}
    r = args.warmup
    for blk in range(n_blocks):
        mode = "fixed" if blk % 2 == 0 else "adaptive"
        for _ in range(ADAPTIVE_BLOCK):
            k = w.k if mode == "fixed" else ctl.next_k()
            if mode == "adaptive":
                chosen[k] = chosen.get(k, 0) + 1
            toks, ms, copy_gbs = one(k, r)
            res[mode][0] += toks * w.layers
            res[mode][1] += ms
            per_round[mode].append((toks * w.layers, ms))
            stalled[mode] += int(copy_gbs is not None and copy_gbs < STALL_FRAC * link_gbs)
            r += 1
    g.close()
    val = {m: v[0] / (v[1] / 1e3) for m, v in res.items()}
    # the same with each mode's median round time (insensitive to the host link's
    # occasional stalls, which land in either mode's blocks at random)
    val_med = {m: statistics.mean(t for t, _ in v) / (statistics.median(ms for _, ms in v) / 1e3)
               for m, v in per_round.items() if v}
    return {"fixed_k": w.k, "k_max": k_max, "choices": choices,
            "rounds_per_arm": {m: len(v) for m, v in per_round.items()}, "block_rounds": ADAPTIVE_BLOCK,
            "fixed_value": val["fixed"], "adaptive_value": val["adaptive"],
            "adaptive_over_fixed": val["adaptive"] / val["fixed"],
            "at_median_round": {"fixed": val_med.get("fixed"), "adaptive": val_med.get("adaptive"),
                                "adaptive_over_fixed": (val_med["adaptive"] / val_med["fixed"])
                                if "fixed" in val_med and "adaptive" in val_med else None},
            "stalled_rounds": stalled, "stall_rule": "copy below %.0f%% of the measured link" % (100 * STALL_FRAC),
            "k_chosen": chosen, "acceptance_estimate": ctl.acceptance(),
            "measured": {"t_step_ms": ctl.t_step, "t_copy_ms": ctl.t_copy, "t_tail_ms": ctl.t_tail,
                         "t_verify_row_ms": ctl.t_row, "link_peak_gbs": link_gbs,
                         "copy_gbs": rate["bytes_per_ms"] / 1e6, "verify_row_chunk_ms": row_chunk_ms}}


def run_adaptive(args, local_rank):
    """--adaptive: the fixed and the controller arm as the headline of the line."""
    import torch

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    w = workload_of(args)
    why = adaptive_skip_reason(w)
    if why:
        raise SystemExit("--adaptive: " + why)
    cmp_ = adaptive_compare(args, device, w, max(2, 2 * args.steps // ADAPTIVE_BLOCK))
    return {"metric": "verified tokens/s/layer", "value": cmp_["adaptive_value"], "unit": "tokens/s/layer",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "dtype": "bf16/int%d->f32" % w.bits, "data": "synthetic (seeded)",
            "config": {"workload": workload_name(w), "schedule": "adaptive draft length", "k_fixed": w.k,
                       "k_max": cmp_["k_max"], "choices": cmp_["choices"]},
            "adaptive": cmp_}


def run_remote(args, local_rank):
    """Remote prefix caching, emulated on one GPU: every layer's packed prefix
    arrives over a slow link paced at --remote-prefix GB/s (real copies through
    vc_quant_kv_stage_groups), then rounds run as usual with the full KV over
    the fast local link.  Compared with shipping the full prefix over the same
    slow link (bytes / rate)."""
    import torch

    import synth
    from verify_compressed_kv_gb300 import runtime as rt

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    w = workload_of(args)
    if w.groups != 1 or w.keep_frac < 1.0:
        raise SystemExit("--remote-prefix runs the single-group workloads without token dropping")
    rate = args.remote_prefix
    rounds = args.warmup + args.steps
    g = build_group(w, w.layers, device, rounds + 2, args.slots or None)
    host = [g.export_packed(l, w.T) for l in range(w.layers)]
    for l in range(w.layers):                     # the draft cache now only exists remotely
        for x in (g.kc, g.ksz, g.vc, g.vsz):
            x[l].zero_()
        g.packed_len[l].zero_()
    comp_bytes = sum(h.numel() * h.element_size() for hs in host for h in hs)
    full_bytes = g.h2d_bytes()
    host_in = [make_round_inputs(w, r, 0, device, w.layers) for r in range(3)]
    inputs = [to_device(x, device) for x in host_in]
    drafts = [x.to(device) for x in round_drafts(w, host_in, rounds + 2, 0)]
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for l in range(w.layers):
        g.stage_packed_remote(l, host[l], w.T, rate, xs)
    xs.synchronize()
    stage_ms = (time.perf_counter() - t0) * 1e3
    t1 = time.perf_counter()
    tl = rt.round_single(g, with_drafts(inputs[0], drafts[0]), cs, xs)
    tl.ev["end"].synchronize()
    first_round_ms = (time.perf_counter() - t1) * 1e3
    first_tokens = g.after_round() * w.layers
    ms, toks = [], 0
    for r in range(1, rounds):
        tl = rt.round_single(g, with_drafts(inputs[r % 3], drafts[r]), cs, xs)
        tl.ev["end"].synchronize()
        t = g.after_round()
        if r >= args.warmup:
            ms.append(tl.ms("start", "end"))
            toks += t * w.layers
    g.close()
    full_ms = full_bytes / (rate * 1e6)
    ttfr = stage_ms + first_round_ms
    return {"metric": "time to the first verified round", "value": ttfr, "unit": "ms", "higher_is_better": False,
            "n_gpus": 1, "data": "synthetic (seeded)",
            "config": {"workload": workload_name(w), "schedule": "remote prefix caching (emulated, one GPU)",
                       "slow_link_gbs": rate},
            "compressed_bytes": comp_bytes, "full_bytes": full_bytes, "bytes_ratio": full_bytes / comp_bytes,
            "stage_ms": stage_ms, "stage_ms_at_rate": comp_bytes / (rate * 1e6), "first_round_ms": first_round_ms,
            "first_round_tokens": first_tokens, "full_prefix_over_slow_link_ms": full_ms,
            "speedup_vs_full_prefix": (full_ms + first_round_ms) / ttfr,
            "steady_value": toks / (sum(ms) / 1e3) if ms else None, "steady_unit": "tokens/s/layer",
            "steady_round_ms": [round(x, 3) for x in ms]}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    return rank, world, local


def combine_rank_results(rows):
    """rows = [(value, e2e, timed_ms)] per rank -> (whole-job value, e2e, max ms).

    Replicas: every rank processed its own requests in its timed region, so
    the job's throughput is all ranks' tokens (value * ms) over the slowest
    rank's time; e2e throughputs add up."""
    t_max = max(r[2] for r in rows)
    value = sum(r[0] * r[2] for r in rows) / t_max
    return value, sum(r[1] for r in rows), t_max


def reduce_over_ranks(value_local, e2e_local, ms_local, world):
    if world <= 1:
        return value_local, e2e_local, ms_local
    import torch
    import torch.distributed as dist
    tt = torch.tensor([value_local, e2e_local, ms_local], dtype=torch.float64)
    vals = [torch.zeros(3, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(vals, tt)
    return combine_rank_results([(float(v[0]), float(v[1]), float(v[2])) for v in vals])


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="llama", choices=["tiny", "mistral", "qwen", "llama", "stagger"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--schedule", default="staggered", choices=["staggered", "lockstep"])
    ap.add_argument("--slots", type=int, default=0,
                    help="verify ring slots per layer (0: as many as the layer's chunks, within a 32 GiB budget)")
    ap.add_argument("--clock-ms", type=int, default=50, help="nvidia-smi sampling interval during the timed region")
    ap.add_argument("--link-peak-gbs", type=float, default=0.0,
                    help="pinned host->device peak in GB/s (default 0: measure it at start-up)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-adaptive", action="store_true",
                    help="leave out the fixed-k vs controller comparison of the default line")
    ap.add_argument("--adaptive", action="store_true",
                    help="compare the fixed draft length with a per-round length chosen by the controller")
    ap.add_argument("--bits", type=int, default=0, choices=[0, 2, 4, 8],
                    help="KIVI code width instead of the workload's own (0: keep it)")
    ap.add_argument("--remote-prefix", type=float, default=0.0, metavar="GBS",
                    help="emulate remote prefix caching: the packed prefix arrives over a link paced at GBS GB/s")
    ap.add_argument("--k-max", type=int, default=60, help="largest draft length of --adaptive (accept takes k + 1 <= 64)")
    ap.add_argument("--k", type=int, default=0, help="draft length instead of the workload's own (0: keep it)")
    ap.add_argument("--rows-only", action="store_true",
                    help="time only the prefill rows (pack, token score / select / gather) of one layer")
    ap.add_argument("--kernel", default="", choices=["", "draft", "verify", "accept"],
                    help="time one kernel alone on one layer (3 warm-up + --calls launches)")
    ap.add_argument("--calls", type=int, default=8, help="timed launches of --kernel")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_setup()
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    elif args.rows_only:
        out = run_rows(args, local) if rank == 0 else None
    elif args.kernel:
        out = run_kernel(args, local) if rank == 0 else None
    elif args.adaptive:
        out = run_adaptive(args, local) if rank == 0 else None
    elif args.remote_prefix > 0:
        out = run_remote(args, local) if rank == 0 else None
    else:
        out = run_ours(args, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
