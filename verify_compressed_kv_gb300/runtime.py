"""Device-side state of a request group and the round driver.

VeriCache (gist.science/paper/2605.17613), Technical Summary:
  * Core Algorithm: draft k tokens with the compressed KV, verify them with
    one pass over the full KV, accept up to the first mismatch (+ the full-KV
    token there), repeat from the last accepted token;
  * Key System Innovations (1), cross-resource staggering: drafting uses HBM,
    verification uses the CPU-GPU link; staggering request groups overlaps
    the two instead of running them in lock-step;
  * Architecture Support: compressed KV in GPU memory, full KV in CPU memory.

Everything here is orchestration: buffers, streams, events and calls into the
C ABI (``_lib``).  Every step of the path runs in the CUDA libraries.

A ``Group`` is one batch of requests with L attention layers.  Per layer it
owns the packed draft cache, the bf16 tail, the pinned chunk-major full-KV
store and the per-request lengths; the group shares a verify slot ring and
workspaces across layers.  Model work outside attention (projections,
sampling) is not part of this path: a round takes its queries, the new
tokens' K/V and the verify logits as inputs (``RoundInputs``).
"""
from __future__ import annotations

import dataclasses
import math
import time

import torch

from . import _lib as vc

GROUP = 32


def _i16(shape, device):
    return torch.empty(shape, dtype=torch.int16, device=device)


@dataclasses.dataclass
class RoundInputs:
    """Per-round device inputs of one group (bf16 tensors are int16 bit views).

    q_draft [L, k, B, Hq, d], kv_cur [2, L, k, B, Hkv, d], q_verify [L, B, k+1, Hq, d],
    kv_new [2, L, B, k+1, Hkv, d], logits fp32 [B, k+1, V], drafts int32 [B, k].
    """
    q_draft: torch.Tensor
    kv_cur: torch.Tensor
    q_verify: torch.Tensor
    kv_new: torch.Tensor
    logits: torch.Tensor
    drafts: torch.Tensor

    @property
    def k(self) -> int:
        """Draft length of this round (<= the group's k)."""
        return int(self.drafts.shape[1])


class LengthBounds:
    """Host-side bounds of a group's lengths, kept from the accepted lengths
    read back every round (each request commits n_acc + 1 tokens a round):
    max_prefix is the longest request's prefix, exactly; max_packed bounds
    packed_len (the tokens packed at load plus every token committed since;
    packed_len is a multiple of 32 at most that)."""

    def __init__(self, B):
        self.committed = torch.zeros(B, dtype=torch.int64)
        self.prefix0 = self.packed0 = 0

    def prefix_from(self, T):
        """The full prefix was (re)written with T tokens a request."""
        self.prefix0 = T
        self.committed.zero_()

    def packed_from(self, T):
        """The draft cache was (re)loaded with T packed tokens a request."""
        self.packed0 = T

    def commit(self, n_acc):
        self.committed += torch.as_tensor(n_acc).to(torch.int64) + 1

    @property
    def max_prefix(self):
        return self.prefix0 + int(self.committed.max())

    @property
    def max_packed(self):
        return self.packed0 + int(self.committed.max())


class Group:
    def __init__(self, B, Hq, Hkv, d, k, bits, V, C, T0, layers=1, extra_tokens=None, n_slots=None,
                 parts_per_chunk=None, softmax_scale=1.0, device="cuda", packed_T0=None,
                 ring_budget_bytes=32 << 30):
        self.B, self.Hq, self.Hkv, self.d, self.k, self.bits, self.V = B, Hq, Hkv, d, k, bits, V
        self.C, self.L = C, layers
        self.device = torch.device(device)
        self.shape = vc.shape(B, Hq, Hkv, d, k=k, bits=bits, softmax_scale=softmax_scale)
        extra = extra_tokens if extra_tokens is not None else 64 * (k + 1)
        self.T_cap = int(math.ceil((T0 + extra) / C) * C)          # host store capacity (tokens)
        self.P0 = T0 if packed_T0 is None else packed_T0             # tokens in the draft cache at start
        self.P_cap = int(math.ceil((self.P0 + extra) / GROUP) * GROUP)
        self.tail_cap = GROUP + k + 1
        if parts_per_chunk is None:
            # the library plans the split from its chunk kernel's occupancy (whole waves)
            parts_per_chunk = vc.vc_verify_attn_parts(self.shape, C)
        self.parts = parts_per_chunk
        dev = self.device
        # ---- draft caches, one per layer
        kcb, kszb, vcb, vszb = vc.vc_quant_packed_bytes(self.shape, self.P_cap)
        self.kc = [torch.zeros(kcb // 4, dtype=torch.int32, device=dev) for _ in range(layers)]
        self.ksz = [torch.zeros(kszb // 2, dtype=torch.int16, device=dev) for _ in range(layers)]
        self.vc = [torch.zeros(vcb // 4, dtype=torch.int32, device=dev) for _ in range(layers)]
        self.vsz = [torch.zeros(vszb // 2, dtype=torch.int16, device=dev) for _ in range(layers)]
        self.tail_k = [torch.zeros((B, Hkv, self.tail_cap, d), dtype=torch.int16, device=dev) for _ in range(layers)]
        self.tail_v = [torch.zeros((B, Hkv, self.tail_cap, d), dtype=torch.int16, device=dev) for _ in range(layers)]
        self.packed_len = [torch.zeros(B, dtype=torch.int32, device=dev) for _ in range(layers)]
        self.tail_len = [torch.zeros(B, dtype=torch.int32, device=dev) for _ in range(layers)]
        # ---- full KV: pinned, chunk-major, one store per layer
        self.n_chunks_cap = self.T_cap // C
        self.chunk_elems = 2 * B * Hkv * C * d
        self.host_kv = [torch.empty(self.n_chunks_cap * self.chunk_elems, dtype=torch.int16, pin_memory=True)
                        for _ in range(layers)]
        self.prefix_len = [torch.zeros(B, dtype=torch.int32, device=dev) for _ in range(layers)]
        self.bounds = LengthBounds(B)
        # ---- verify rings (one per layer) + workspaces.  A round prefetches every
        # layer's first chunks while the group drafts, so the link is busy from the
        # start of the round; by default each ring holds all of its layer's chunks
        # when the rings of all layers fit the HBM budget.
        if n_slots is None:
            per_layer = ring_budget_bytes // (layers * self.chunk_elems * 2)
            n_slots = int(max(2, min(self.n_chunks_cap, per_layer)))
        self.n_slots = n_slots                 # per layer
        self.ring = [_i16(n_slots * self.chunk_elems, dev) for _ in range(layers)]
        # sized for every draft length a round may use (1 .. k): the needs are not monotone in k
        self.ws_verify_bytes = max(vc.vc_verify_attn_workspace_size(
            vc.shape(B, Hq, Hkv, d, k=kk, bits=bits, softmax_scale=softmax_scale), self.parts) for kk in range(1, k + 1))
        self.ws_verify = torch.zeros(self.ws_verify_bytes, dtype=torch.uint8, device=dev)
        self.ws_draft_bytes = vc.vc_draft_attn_workspace_size(self.shape, self.P_cap)
        self.ws_draft = torch.zeros(self.ws_draft_bytes, dtype=torch.uint8, device=dev)
        self.ws_accept_bytes = max(vc.vc_accept_workspace_size(B, kk, V) for kk in range(1, k + 1))
        self.ws_accept = torch.zeros(self.ws_accept_bytes, dtype=torch.uint8, device=dev)
        self.pipes = [vc.vc_verify_pipeline_create(n_slots) for _ in range(layers)]
        self.launches = 0                      # kernels launched through this group
        # ---- per-round outputs
        self.draft_out = _i16((B, Hq, d), dev)
        self.verify_out = _i16((B, k + 1, Hq, d), dev)
        self.n_acc = torch.zeros(B, dtype=torch.int32, device=dev)
        self.next_tok = torch.zeros(B, dtype=torch.int32, device=dev)
        self.n_acc_host = torch.zeros(B, dtype=torch.int32, pin_memory=True)
        self._shapes = {}

    @property
    def max_prefix(self):
        return self.bounds.max_prefix

    def shape_k(self, k):
        """Shape struct of a round drafting k <= self.k tokens (buffers and
        workspaces sized for self.k fit every smaller k)."""
        if k == self.k:
            return self.shape
        if not 1 <= k <= self.k:
            raise ValueError(f"draft length {k} outside [1, {self.k}]")
        if k not in self._shapes:
            s = self.shape
            self._shapes[k] = vc.shape(self.B, self.Hq, self.Hkv, self.d, k=k, bits=self.bits,
                                       softmax_scale=s.softmax_scale)
        return self._shapes[k]

    def verify_out_k(self, k):
        """verify_out viewed as [B, k+1, Hq, d] (its leading elements)."""
        n = self.B * (k + 1) * self.Hq * self.d
        return self.verify_out.view(-1)[:n].view(self.B, k + 1, self.Hq, self.d)

    def close(self):
        for p in self.pipes:
            vc.vc_verify_pipeline_destroy(p)
        self.pipes = []

    # ---------------------------------------------------------------- prefill
    def load_prefix(self, layer, K, V, stream=None):
        """Prefix K/V of a layer, bf16 [B, Hkv, T0, d] int16 tensors on the device:
        quantise + pack into the draft cache and copy into the pinned store."""
        T0 = K.shape[2]
        assert T0 % GROUP == 0 and T0 <= self.P_cap
        vc.vc_quant_kv_pack(self.shape, T0, self.P_cap, K, V, self.kc[layer], self.ksz[layer], self.vc[layer],
                            self.vsz[layer], stream)
        self.packed_len[layer].fill_(T0)
        self.tail_len[layer].zero_()
        self.write_store(layer, K, V)
        self.bounds.packed_from(T0)

    def load_packed_only(self, layer, K, V, stream=None):
        """Draft cache from an already-compressed (e.g. token-dropped) prefix."""
        T = K.shape[2]
        vc.vc_quant_kv_pack(self.shape, T, self.P_cap, K, V, self.kc[layer], self.ksz[layer], self.vc[layer],
                            self.vsz[layer], stream)
        self.packed_len[layer].fill_(T)
        self.tail_len[layer].zero_()
        self.bounds.packed_from(T)

    # ---------------------------------------------------------------- remote prefix (emulated)
    def export_packed(self, layer, T):
        """The packed groups of tokens [0, T) of a layer, in pinned host memory:
        the store a remote prefix cache would hold (kc, ksz, vc, vsz arrays laid
        out like the device ones with T/32 groups per (request, KV head))."""
        ng, NGc, BH = T // GROUP, self.P_cap // GROUP, self.B * self.Hkv
        out = []
        for x in (self.kc, self.ksz, self.vc, self.vsz):
            v = x[layer].view(BH, NGc, -1)[:, :ng].contiguous()
            out.append(v.cpu().pin_memory())
        return out

    def stage_packed_remote(self, layer, host, T, link_gbs, stream, groups_per_copy=32):
        """Stream a remote packed store into the layer's draft cache over an
        emulated slow link: the copies go out in pieces of `groups_per_copy`
        groups, each issued no earlier than the time the link would have
        delivered the bytes before it at `link_gbs` GB/s (host pacing; the copy
        engine itself runs at the local link's speed).  Returns the host wall
        time at which the last piece was issued; packed_len is set on `stream`
        after the last piece."""
        ng = T // GROUP
        per_group = sum(h[0, 0].numel() * h.element_size() for h in host) * self.B * self.Hkv
        t0 = time.perf_counter()
        sent = 0
        for g0 in range(0, ng, groups_per_copy):
            g1 = min(ng, g0 + groups_per_copy)
            wait = sent / (link_gbs * 1e9) - (time.perf_counter() - t0)
            if wait > 0:
                time.sleep(wait)
            vc.vc_quant_kv_stage_groups(self.shape, host[0], host[1], host[2], host[3], ng, g0, g1, self.P_cap,
                                        self.kc[layer], self.ksz[layer], self.vc[layer], self.vsz[layer], stream)
            sent += (g1 - g0) * per_group
        wait = sent / (link_gbs * 1e9) - (time.perf_counter() - t0)
        if wait > 0:
            time.sleep(wait)
        with torch.cuda.stream(stream):
            self.packed_len[layer].fill_(T)
            self.tail_len[layer].zero_()
        self.bounds.packed_from(T)
        return time.perf_counter() - t0

    def write_store(self, layer, K, V):
        """Full prefix K/V [B, Hkv, T, d] (device or host) -> pinned chunk-major store."""
        T = K.shape[2]
        st = self.host_kv[layer].view(self.n_chunks_cap, 2, self.B, self.Hkv, self.C, self.d)
        for c in range((T + self.C - 1) // self.C):
            n = min(self.C, T - c * self.C)
            st[c, 0, :, :, :n].copy_(K[:, :, c * self.C:c * self.C + n])
            st[c, 1, :, :, :n].copy_(V[:, :, c * self.C:c * self.C + n])
        self.prefix_len[layer].fill_(T)
        self.bounds.prefix_from(T)

    # ---------------------------------------------------------------- the round's steps
    def prefetch(self, layer, copy_stream):
        vc.vc_verify_prefetch(self.pipes[layer], self.shape, self.host_kv[layer], self.C, self.max_prefix, self.T_cap,
                              self.ring[layer], copy_stream)

    def prefetch_all(self, copy_stream):
        """Every layer's first n_slots chunks, in layer order, on the copy stream."""
        for layer in range(self.L):
            self.prefetch(layer, copy_stream)

    def draft_step(self, inp: RoundInputs, layer: int, step: int, stream, chained=False):
        """chained: the previous work on `stream` is another draft call, so
        this one may start while that one finishes (VC_DRAFT_CHAINED)."""
        # packed_len is a multiple of 32 no larger than the host bound: the
        # partition then covers the packed groups, not the cache's capacity
        max_packed = min(self.P_cap, self.bounds.max_packed // GROUP * GROUP)
        vc.vc_draft_attn(self.shape, inp.q_draft[layer, step], inp.kv_cur[0, layer, step], inp.kv_cur[1, layer, step],
                         self.kc[layer], self.ksz[layer], self.vc[layer], self.vsz[layer], self.packed_len[layer],
                         max_packed, self.P_cap, self.tail_k[layer], self.tail_v[layer], self.tail_len[layer],
                         self.tail_cap, step, self.draft_out, self.ws_draft, self.ws_draft_bytes, stream,
                         flags=vc.VC_DRAFT_CHAINED if chained else 0)
        self.launches += 1                     # stream CTAs, tail CTAs and the combine: one grid

    def verify(self, inp: RoundInputs, layer: int, compute_stream, copy_stream):
        vc.vc_verify_attn_streamed(self.pipes[layer], self.shape_k(inp.k), inp.q_verify[layer], self.host_kv[layer],
                                   self.C, self.max_prefix, self.T_cap, self.prefix_len[layer], self.ring[layer],
                                   inp.kv_new[0, layer],
                                   inp.kv_new[1, layer], self.verify_out_k(inp.k), self.parts, self.ws_verify,
                                   self.ws_verify_bytes, compute_stream, copy_stream)
        self.launches += self.chunks() + 1     # one kernel per chunk, then the new-token block + merge

    def decode_full_kv(self, q1, kv1, out1, layer, compute_stream, copy_stream):
        """One plain decoding step over the full KV (the baseline the pages
        compare against): the same streamed verify path with one row (k = 0).
        q1 [B, 1, Hq, d], kv1 [2, B, 1, Hkv, d], out1 [B, 1, Hq, d]."""
        if not hasattr(self, "_shape0"):
            self._shape0 = vc.shape(self.B, self.Hq, self.Hkv, self.d, k=0, bits=self.bits,
                                    softmax_scale=self.shape.softmax_scale)
            self._ws0_bytes = vc.vc_verify_attn_workspace_size(self._shape0, self.parts)
            self._ws0 = torch.zeros(self._ws0_bytes, dtype=torch.uint8, device=self.device)
        vc.vc_verify_attn_streamed(self.pipes[layer], self._shape0, q1, self.host_kv[layer], self.C, self.max_prefix,
                                   self.T_cap, self.prefix_len[layer], self.ring[layer], kv1[0], kv1[1], out1, self.parts, self._ws0,
                                   self._ws0_bytes, compute_stream, copy_stream)
        self.launches += self.chunks() + 1

    def accept(self, inp: RoundInputs, stream):
        vc.vc_accept(self.B, inp.k, self.V, inp.logits, inp.drafts, self.n_acc, self.next_tok, None,
                     self.ws_accept, self.ws_accept_bytes, stream)
        self.launches += 1

    def commit(self, inp: RoundInputs, stream):
        sh = self.shape_k(inp.k)
        for l in range(self.L):
            vc.vc_verify_commit(sh, inp.kv_new[0, l], inp.kv_new[1, l], self.n_acc, self.prefix_len[l],
                                self.host_kv[l], self.C, self.T_cap, stream)
            vc.vc_quant_kv_append(sh, inp.kv_new[0, l], inp.kv_new[1, l], self.n_acc, self.tail_k[l],
                                  self.tail_v[l], self.tail_len[l], self.tail_cap, self.kc[l], self.ksz[l],
                                  self.vc[l], self.vsz[l], self.packed_len[l], self.P_cap, stream)
            self.launches += 4                 # commit, commit lengths, append, append lengths

    def prefetch_bytes(self):
        """Bytes prefetch_all() moves: the first min(n_slots, chunks) chunks of every layer."""
        total = 0
        for c in range(min(self.n_slots, self.chunks())):
            total += 2 * self.B * self.Hkv * min(self.C, self.max_prefix - c * self.C) * self.d * 2
        return total * self.L

    def chunks(self):
        return (self.max_prefix + self.C - 1) // self.C

    def h2d_bytes(self):
        """Full-KV bytes one verify pass moves over the link (all layers)."""
        return self.L * 2 * self.B * self.Hkv * self.max_prefix * self.d * 2

    def read_back(self, stream):
        """Device -> host copy of the accepted lengths (the round's result)."""
        with torch.cuda.stream(stream):
            self.n_acc_host.copy_(self.n_acc, non_blocking=True)

    def after_round(self):
        """Host bookkeeping once the read-back has landed."""
        n = self.n_acc_host
        self.bounds.commit(n)
        if self.max_prefix > self.T_cap:
            raise RuntimeError(f"the group's full-KV store holds {self.T_cap} tokens a request, the prefix reached "
                               f"{self.max_prefix}: size extra_tokens for every round the group makes")
        return int(n.sum()) + self.B          # tokens produced this round


class Timeline:
    """CUDA events (with timing) recorded on the streams of one round."""

    def __init__(self):
        self.ev = {}

    def mark(self, name, stream):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        self.ev[name] = e
        return e

    def ms(self, a, b):
        return self.ev[a].elapsed_time(self.ev[b])


def _inputs_first(copy_in, xs, cs):
    """The round's host inputs over the link ahead of its bulk full-KV stream:
    copy_in(stream) enqueues their copies on the copy stream, the drafting
    waits for them."""
    if copy_in is None:
        return
    copy_in(xs)
    ev = torch.cuda.Event()
    ev.record(xs)
    cs.wait_event(ev)


def round_single(g: Group, inp: RoundInputs, cs, xs, tl: Timeline | None = None, ready=None, copy_in=None):
    """One round of one group: the first chunks of every layer's full KV start
    streaming while the group drafts (prefix chunks do not depend on the
    drafts), then verify, accept, commit.  `ready`: an event the round's inputs
    wait for (e.g. their copy from host memory on another stream); the full-KV
    stream does not.  `copy_in(stream)`: enqueue the copies of the round's inputs
    from host memory; they go on the copy stream ahead of the full KV, and the
    drafting waits for them.  Returns the round's timeline; call
    g.after_round() after syncing."""
    tl = tl or Timeline()
    tl.mark("start", cs)
    xs.wait_event(tl.ev["start"])
    tl.mark("copy_start", xs)
    _inputs_first(copy_in, xs, cs)
    g.prefetch_all(xs)
    tl.mark("prefetch_end", xs)            # the first slots' copies: they never wait for a slot
    if ready is not None:
        cs.wait_event(ready)
    tl.mark("draft_start", cs)
    for i in range(inp.k):
        for l in range(g.L):
            g.draft_step(inp, l, i, cs, chained=i + l > 0)
    tl.mark("draft_end", cs)
    for l in range(g.L):
        g.verify(inp, l, cs, xs)
    tl.mark("copy_end", xs)
    tl.mark("verify_end", cs)
    g.accept(inp, cs)
    tl.mark("commit_start", cs)
    g.commit(inp, cs)
    tl.mark("commit_end", cs)
    cs.wait_event(tl.ev["copy_end"])
    g.read_back(cs)
    tl.mark("end", cs)
    return tl


def round_staggered(X: Group, Y: Group, inp_x: RoundInputs, inp_y: RoundInputs, cs, xs, tl: Timeline | None = None,
                    ready=None, copy_in=None):
    """Cross-resource staggering: X drafts (HBM) while Y's full KV streams over
    the link and Y verifies, accepts and commits.  Roles swap every round.
    `ready` and `copy_in` as in round_single."""
    tl = tl or Timeline()
    tl.mark("start", cs)
    xs.wait_event(tl.ev["start"])
    tl.mark("copy_start", xs)
    _inputs_first(copy_in, xs, cs)
    Y.prefetch_all(xs)
    if ready is not None:
        cs.wait_event(ready)
    tl.mark("draft_start", cs)
    for i in range(inp_x.k):
        for l in range(X.L):
            X.draft_step(inp_x, l, i, cs, chained=i + l > 0)
    tl.mark("draft_end", cs)
    for l in range(Y.L):
        Y.verify(inp_y, l, cs, xs)
    tl.mark("copy_end", xs)
    tl.mark("verify_end", cs)
    Y.accept(inp_y, cs)
    tl.mark("commit_start", cs)
    Y.commit(inp_y, cs)
    tl.mark("commit_end", cs)
    cs.wait_event(tl.ev["copy_end"])
    Y.read_back(cs)
    tl.mark("end", cs)
    return tl


def round_lockstep(groups, inps, cs, xs, tl: Timeline | None = None):
    """The comparison schedule: every group drafts, then every group verifies;
    no transfer starts before drafting ends."""
    tl = tl or Timeline()
    tl.mark("start", cs)
    tl.mark("draft_start", cs)
    first = True
    for g, inp in zip(groups, inps):
        for i in range(inp.k):
            for l in range(g.L):
                g.draft_step(inp, l, i, cs, chained=not first)
                first = False
    tl.mark("draft_end", cs)
    xs.wait_event(tl.ev["draft_end"])
    tl.mark("copy_start", xs)
    for g, inp in zip(groups, inps):
        for l in range(g.L):
            g.verify(inp, l, cs, xs)
        g.accept(inp, cs)
        g.commit(inp, cs)
    tl.mark("copy_end", xs)
    tl.mark("verify_end", cs)
    cs.wait_event(tl.ev["copy_end"])
    for g in groups:
        g.read_back(cs)
    tl.mark("end", cs)
    return tl
