#!/usr/bin/env python
"""Throughput of the tree-verification step (Medusa / EAGLE) on GB300.

One step = one pass of the whole hot path over one batch of synthetic
inputs resident in HBM.  The default workload is 70B-shaped batched serving
(batch 64, 64 query / 8 KV heads, head_dim 128, bf16, prefix 4096, a 32-node
static tree of 4 levels, vocabulary 128256): static tree build -> tree
attention (one layer) -> greedy acceptance -> batched KV commit.  Other
workloads: --workload {tiny_exact, vicuna7b_medusa, llama8b_eagle2,
llama70b_serving, long_context}; the default run also reports the full step
rate of each of the other four under "workloads".

Timing: the K steps are captured once as a CUDA graph; the graph is replayed
back to back for at least --min-seconds (so the clock sampler sees the GPU
under load) and the median replay, divided by K, is the step time.

Prints one JSON line (rank 0).  N > 1 (torchrun) runs independent replicas
(no collective on the data path; weak scaling).  ``--impl reference`` times
the CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

if "reference" in sys.argv and "--impl" in sys.argv:
    # the CPU oracle runs on one core; pin the numeric libraries before
    # numpy loads them so the reported core count is the one used
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = "1"

import numpy as np  # noqa: E402

DEFAULT = "llama70b_serving"
L2_BYTES = 129 * 1024 * 1024

# DRAM bytes (read + write) per call of a stage, from one ncu capture of
# that stage's kernel at the workload's shape, valid only while the kernel
# source is the one the counters were taken on: (source, sha256 prefix,
# bytes) keyed by (workload, stage).
NCU_TRAFFIC = {
    # attn_tc2_kernel, 70B shape at batch 16 (one quarter of the workload's
    # sequences; traffic grows with the sequences): (286,022,272 read +
    # 6,765,184 written, mean of two launches) x 4, from one ncu capture
    # (taken on this code; the source has changed since only in comments)
    ("llama70b_serving", "tree_attn"): ("csrc/attn_tc2.cu", "178217b7f9f1ce91", 1171149824),
}


def measured_traffic(workload: str, stage: str):
    import hashlib
    ent = NCU_TRAFFIC.get((workload, stage))
    if not ent:
        return None
    path = os.path.join(ROOT, "tree_speculative_decoding_attn_gb300", ent[0])
    with open(path, "rb") as f:
        return ent[2] if hashlib.sha256(f.read()).hexdigest()[:16] == ent[1] else None


def wgemm_launches(M: int, K: int, G: int, rows: int, sms: int) -> int:
    """Kernel launches of one weight-streaming GEMM of rows <= 256: the GEMM,
    plus the stream-K fixup when a tile's K chunks span two CTAs (the
    library's plan: 16..128 activation rows use 256-row W tiles, 256 rows
    128-row tiles; 64-wide K chunks; one contiguous unit range per CTA)."""
    km = 256 if rows <= 128 else 128
    nk, tiles = K // 64, -(-M // km) * G
    units = tiles * nk
    ctas = min(units, sms)
    cta_of = lambda x: ((x + 1) * ctas - 1) // units
    return 1 + any(cta_of(t * nk) != cta_of(t * nk + nk - 1) for t in range(tiles))


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0])); mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# the GPU step
# ----------------------------------------------------------------------------
class GpuStep:
    """Device buffers of one workload and the launches of one verify step."""

    def __init__(self, name: str, device):
        import torch
        from tree_speculative_decoding_attn_gb300 import specverify as sv
        from tree_speculative_decoding_attn_gb300 import synth
        self.torch, self.sv, self.synth = torch, sv, synth
        w = self.w = synth.WORKLOADS[name]
        self.name = name
        dev = self.dev = device
        self.sms = torch.cuda.get_device_properties(dev).multi_processor_count
        bf = torch.bfloat16
        tdt = self.tdt = bf if w.dtype == "bf16" else torch.float32
        cu = lambda x, dt=None: (torch.from_numpy(np.ascontiguousarray(x)).to(dt) if dt else
                                 torch.from_numpy(np.ascontiguousarray(x))).to(dev)
        i32 = lambda *s: torch.zeros(s, dtype=torch.int32, device=dev)
        B, N, Hq, Hkv, D, V = w.batch, w.n_nodes, w.hq, w.hkv, w.head_dim, w.vocab
        self.prefix = synth.prefix_lengths(w)
        self.max_prefix = int(self.prefix.max())
        self.s_max = self.max_prefix + 64
        self.stages = []          # (name, fn, launches, algorithmic bytes or None)
        self.h2d = []             # (pinned host copy, attribute name) copied each end-to-end step
        # tree
        if w.tree == "dynamic":
            dk = w.dynamic
            if dk.get("draft"):
                self._eagle_setup()         # the pool is drafted on the GPU each step
            else:
                par, tok, conf = synth.candidate_pool(w.seed, B, dk["k"], dk["frontier"], dk["rounds"], V)
                self.pool = [cu(par), cu(tok), cu(conf)]
            self.path_cap = dk["rounds"] + 2
            self.shape = None
        else:
            self.shape = synth.tree_shape(w)
            self.path_cap = self.shape.n_levels + 1
            self.parents = cu(self.shape.parents)
            self.rank = cu(self.shape.rank)
            self.parents_b = cu(np.broadcast_to(self.shape.parents, (B, N)).copy())
        self.root = cu(synth.root_tokens(w))
        self.d_prefix = cu(self.prefix)
        self.tok, self.depth, self.pos = i32(B, N), i32(B, N), i32(B, N)
        self.fc, self.ns, self.par_out = i32(B, N), i32(B, N), i32(B, N)
        self.anc = torch.zeros((B, N), dtype=torch.int64, device=dev)
        self.status = i32(1)
        # attention inputs
        q, kc, vc, kt, vt = synth.attention_inputs(w, self.prefix, s_max=self.s_max)
        self.q, self.kc, self.vc, self.kt, self.vt = (cu(x, tdt) for x in (q, kc, vc, kt, vt))
        del q, kc, vc, kt, vt
        self.out = torch.empty((B, N, Hq, D), dtype=tdt, device=dev)
        # split count from the host-known prefix lengths (matters for ragged batches)
        self.splits = sv.tree_attn_plan_splits(tdt, B, N, Hq, Hkv, D, self.prefix)
        wsb = sv.tree_attn_workspace_bytes(tdt, B, N, Hq, Hkv, D, self.max_prefix, self.splits)
        self.ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
        self.attn_launches = 2 if wsb > 0 else 1
        esz = 2 if tdt == bf else 4
        # algorithmic bytes: every prefix and tree K/V row once, Q in, O out
        self.attn_bytes = int(Hkv * D * 2 * esz * (int(self.prefix.sum()) + B * N) + 2 * B * N * Hq * D * esz)
        self.attn_flops = int(4 * N * (Hq // Hkv) * D * Hkv * (int(self.prefix.sum()) + B * N))
        # acceptance outputs
        self.acc_len, self.acc_path, self.bonus = i32(B), i32(B, self.path_cap), i32(B)
        self.new_prefix = i32(B)
        # per-step inputs for the end-to-end leg: this pass's tree Q/K/V and
        # the per-sequence scalars
        for nm in ("q", "kt", "vt", "d_prefix", "root"):
            self.e2e_input(nm)
        self.d2h_names = ["acc_len", "acc_path", "bonus", "new_prefix"]  # results read back per step

        if w.medusa:
            self._medusa_stages(cu)
        else:
            self._static_or_dynamic_build(cu)
            self.logits_bytes_row = V * (2 if w.dtype == "bf16" else 4)
            lg = synth.target_logits(w.seed, B, N, V, w.logit_std, w.dtype == "bf16")
            if w.planted and w.tree != "dynamic":
                cand = synth.candidate_tokens(w.seed, B, self.shape.n_levels, max(w.caps or (2,)), V)
                synth.plant_agreement(w.seed, lg, self.shape.parents, self.shape.level,
                                      synth.node_tokens_from_table(self.shape, cand, synth.root_tokens(w)),
                                      bf16=w.dtype == "bf16")
            elif w.planted:
                # plant on the tree the GPU builds from the (drafted) pool (deterministic)
                for nm, fn, _, _ in self.stages:
                    fn()
                    if nm == "build_tree":
                        break
                torch.cuda.synchronize()
                synth.plant_agreement(w.seed, lg, self.par_out.cpu().numpy(), self.depth.cpu().numpy(),
                                      self.tok.cpu().numpy(), bf16=True)
            self.logits = cu(lg, tdt)
            del lg
        self._attn_stage()
        # the fused LM head + acceptance (statistics epilogue) is an entry point
        # of its own; the step keeps the LM head and the acceptance apart,
        # which measured faster at the Vicuna shape (see the design notes)
        self.fused_accept = False
        if w.medusa:
            self._lm_head_stage(cu)
        self._accept_commit_stages()

    # ---- stages ----------------------------------------------------------
    def _medusa_stages(self, cu):
        torch, sv, synth, w = self.torch, self.sv, self.synth, self.w
        m = w.medusa
        B, K, d, V, s = w.batch, m["heads"], m["hidden"], w.vocab, m["topk"]
        h, w1, w2, wlm = synth.medusa_inputs(w)
        bf = torch.bfloat16
        self.h = cu(h, bf)
        self.w1, self.w2, self.wlm = cu(w1, bf), cu(w2, bf), cu(wlm, bf)
        del w1, w2, wlm
        self.z = torch.empty((B, K, d), dtype=bf, device=self.dev)
        self.head_logits = torch.empty((B, K, V), dtype=torch.float32, device=self.dev)
        self.heads_ws = torch.empty(max(sv.spec_medusa_heads_workspace_bytes(B, K, d, V), 16), dtype=torch.uint8,
                                    device=self.dev)
        self.cand = torch.empty((B, K, s), dtype=torch.int32, device=self.dev)
        self.e2e_input("h")
        # algorithmic bytes: both weight matrices once, h in, z out (bf16), logits out
        heads_bytes = 2 * K * d * d + 2 * K * V * d + 2 * B * d + 2 * B * K * d + 4 * B * K * V
        self.stages.append(("medusa_heads", lambda: sv.spec_medusa_heads(
            self.h, self.w1, None, self.w2, self.z, self.head_logits, workspace=self.heads_ws,
            dev_status=self.status), wgemm_launches(d, d, K, B, self.sms) + wgemm_launches(V, d, K, B, self.sms),
            heads_bytes))  # W1 then W2, each with its fixup
        self.stages.append(("topk", lambda: sv.spec_topk(self.head_logits, s, self.cand), 1, 4 * B * K * V))
        self.stages.append(("build_tree", lambda: sv.spec_build_tree(
            self.parents, self.rank, self.cand, self.root, self.d_prefix, self.tok, self.depth, self.pos, self.anc,
            self.fc, self.ns, self.status), 1, None))

    def _eagle_setup(self):
        """EAGLE-2 drafting on the GPU: random draft-layer weights of the
        target's shape (drawn on the device from a seeded generator), the
        draft layer's prefix cache, and a pool grown by `rounds` drafting
        rounds from the root: k children per frontier node, the next frontier
        the `frontier` new nodes of highest path value."""
        torch, sv, w = self.torch, self.sv, self.w
        dk, dr = w.dynamic, w.dynamic["draft"]
        dev, bf = self.dev, torch.bfloat16
        B, hq, hkv, D, V = w.batch, w.hq, w.hkv, w.head_dim, w.vocab
        d, ffn, k, F, R = hq * D, dr["ffn"], dk["k"], dk["frontier"], dk["rounds"]
        M = 1 + k + (R - 1) * F * k
        gen = torch.Generator(device=dev).manual_seed(w.seed + 77)
        rnd = lambda *shape, std=1.0, mean=0.0: (torch.randn(shape, generator=gen, device=dev) * std + mean).to(bf)
        sd = dr["w_std"]
        self.eagle_w = dict(fc=rnd(d, 2 * d, std=sd), ln1=rnd(d, std=0.05, mean=1.0), qkv=rnd((hq + 2 * hkv) * D, d, std=sd),
                            o=rnd(d, hq * D, std=sd), ln2=rnd(d, std=0.05, mean=1.0), gate_up=rnd(2, ffn, d, std=sd),
                            down=rnd(d, ffn, std=sd), lnf=rnd(d, std=0.05, mean=1.0), lm=rnd(V, d, std=sd),
                            emb=rnd(V, d))
        S = self.s_max
        self.e_kp, self.e_vp = rnd(B, hkv, S, D), rnd(B, hkv, S, D)
        self.e_kn = torch.zeros((B, hkv, M, D), dtype=bf, device=dev)
        self.e_vn = torch.zeros_like(self.e_kn)
        self.e_feat = torch.zeros((B, M + 1, d), dtype=bf, device=dev)
        self.e_feat[:, M] = rnd(B, d)
        root = torch.from_numpy(self.synth.root_tokens(w)).to(dev)
        i32 = lambda *sh: torch.zeros(sh, dtype=torch.int32, device=dev)
        self.e_par0 = torch.full((B, M), -1, dtype=torch.int32, device=dev)
        self.e_tok0 = i32(B, M)
        self.e_tok0[:, 0] = root
        self.e_conf0 = torch.zeros((B, M), dtype=torch.float32, device=dev)
        self.e_conf0[:, 0] = 1.0
        self.e_cnt0 = torch.ones(B, dtype=torch.int32, device=dev)
        self.pool = [self.e_par0.clone(), self.e_tok0.clone(), self.e_conf0.clone()]
        self.e_val, self.e_cnt = self.e_conf0.clone(), self.e_cnt0.clone()
        self.e_front = [i32(B, 1), i32(B, F), i32(B, F)]
        self.e_ws = torch.empty(sv.spec_eagle_round_workspace_bytes(B, F, d, hq, hkv, D, ffn, V, S, self.max_prefix),
                                dtype=torch.uint8, device=dev)
        self.e_rounds = R
        # this layer's weight and cache bytes streamed per round (algorithmic)
        self.eagle_round_bytes = 2 * (d * 2 * d + (hq + 2 * hkv) * D * d + d * hq * D + 2 * ffn * d + d * ffn + V * d) \
            + hkv * D * 2 * 2 * (int(self.prefix.sum()))

    def eagle_launches(self):
        """Kernels of the drafting rounds: per round the six GEMMs (+ their
        fixups), nine row kernels, the tree build, attention + merge and the
        two expansion kernels."""
        w, sms = self.w, self.sms
        hq, hkv, D, ffn, V = w.hq, w.hkv, w.head_dim, w.dynamic["draft"]["ffn"], w.vocab
        d = hq * D
        n = 0
        for r in range(self.e_rounds):
            R = w.batch * (1 if r == 0 else w.dynamic["frontier"])
            n += sum(wgemm_launches(M, K, G, R, sms) for M, K, G in
                     ((d, 2 * d, 1), ((hq + 2 * hkv) * D, d, 1), (d, hq * D, 1), (ffn, d, 2), (d, ffn, 1), (V, d, 1)))
            n += 9 + 1 + 2 + 2
        return n

    def _eagle_rounds(self):
        sv, w = self.sv, self.w
        par, tok, conf = self.pool
        par.copy_(self.e_par0); tok.copy_(self.e_tok0); conf.copy_(self.e_conf0)
        self.e_val.copy_(self.e_conf0); self.e_cnt.copy_(self.e_cnt0)
        front = self.e_front[0]
        for r in range(self.e_rounds):
            nxt = self.e_front[1 + (r % 2)]
            sv.spec_eagle_round(self.eagle_w, self.e_kp, self.e_vp, self.d_prefix, self.max_prefix, self.e_kn,
                                self.e_vn, self.e_feat, front, r, w.dynamic["k"], w.temperature, par, tok, conf,
                                self.e_val, self.e_cnt, nxt, workspace=self.e_ws, dev_status=self.status)
            front = nxt

    def _static_or_dynamic_build(self, cu):
        sv, synth, w = self.sv, self.synth, self.w
        if w.tree == "dynamic" and w.dynamic.get("draft"):
            self.stages.append(("eagle_draft", self._eagle_rounds, self.eagle_launches(),
                                self.eagle_round_bytes * self.e_rounds))
        if w.tree == "dynamic":
            par, tok, conf = self.pool
            self.stages.append(("build_tree", lambda: sv.spec_build_tree_dynamic(
                par, tok, conf, self.d_prefix, self.tok, self.par_out, self.depth, self.pos, self.anc, self.fc,
                self.ns, None, None, self.status), 1, None))
        else:
            s = max(w.caps) if w.caps else 2
            self.cand = cu(synth.candidate_tokens(w.seed, w.batch, self.shape.n_levels, s, w.vocab))
            self.stages.append(("build_tree", lambda: sv.spec_build_tree(
                self.parents, self.rank, self.cand, self.root, self.d_prefix, self.tok, self.depth, self.pos,
                self.anc, self.fc, self.ns, self.status), 1, None))

    def _attn_stage(self):
        sv = self.sv
        self.stages.append(("tree_attn", lambda: sv.tree_attn_verify(
            self.q, self.kc, self.vc, self.kt, self.vt, self.d_prefix, self.anc, self.out, self.max_prefix,
            num_splits=self.splits, workspace=self.ws, dev_status=self.status), self.attn_launches, self.attn_bytes))

    def _lm_head_stage(self, cu):
        torch, sv, synth, w = self.torch, self.sv, self.synth, self.w
        B, N, V, d = w.batch, w.n_nodes, w.vocab, w.medusa["hidden"]
        g = synth.stream(w.seed, "tree_hidden")
        self.hid = cu(synth.gaussian(g, (B * N, d), 1.0, True), torch.bfloat16)
        self.logits = torch.empty((B, N, V), dtype=torch.float32, device=self.dev)
        self.logits_bytes_row = V * 4
        self.e2e_input("hid")
        if self.fused_accept:  # the LM head runs inside the lm_head_accept stage
            self.lm_ws = torch.empty(max(sv.spec_lm_head_accept_workspace_bytes(B, N, d, V), 16),
                                     dtype=torch.uint8, device=self.dev)
            return
        self.lm_ws = torch.empty(max(sv.spec_lm_head_workspace_bytes(B * N, d, V), 16), dtype=torch.uint8,
                                 device=self.dev)
        self.stages.append(("lm_head", lambda: sv.spec_lm_head(self.hid, self.wlm, self.logits.view(B * N, V),
                                                               dev_status=self.status, workspace=self.lm_ws),
                            wgemm_launches(V, d, 1, B * N, self.sms),
                            2 * V * d + 2 * B * N * d + 4 * B * N * V))

    def lm_head_logits(self):
        """The unfused LM head's float32 logits of this step's tree rows
        (reference for tests of the fused stage)."""
        w = self.w
        B, N, V, d = w.batch, w.n_nodes, w.vocab, w.medusa["hidden"]
        self.sv.spec_lm_head(self.hid, self.wlm, self.logits.view(B * N, V), dev_status=self.status)
        return self.logits

    def _accept_commit_stages(self):
        sv, w = self.sv, self.w
        mode = {"greedy": sv.GREEDY, "typical": sv.TYPICAL, "reject": sv.REJECT}[w.accept]
        parents = self.par_out if w.tree == "dynamic" else self.parents_b
        self.step_counter = 0
        if self.fused_accept:
            B, N, V, d = w.batch, w.n_nodes, w.vocab, w.medusa["hidden"]
            # the GEMM (+ its stream-K fixup) and the fold kernel
            launches = wgemm_launches(V, d, 1, B * N, self.sms) + 1
            self.stages.append(("lm_head_accept", lambda: sv.spec_lm_head_accept(
                mode, self.hid.view(B, N, d), self.wlm, self.tok, parents, self.fc, self.ns, self.acc_len,
                self.acc_path, self.bonus, temperature=w.temperature, eps=w.eps, delta=w.delta,
                dev_status=self.status, workspace=self.lm_ws), launches, 2 * V * d + 2 * B * N * d))
            self.stages.append(("kv_commit", lambda: sv.kv_commit(
                self.kc, self.vc, self.kt, self.vt, self.acc_len, self.acc_path, self.d_prefix, self.new_prefix,
                self.status), 1, None))
        else:
            # acceptance and the commit of the accepted path in one launch
            self.stages.append(("accept_commit", lambda: sv.spec_accept_commit(
                mode, self.logits, self.tok, parents, self.fc, self.ns, self.acc_len, self.acc_path, self.bonus,
                self.kc, self.vc, self.kt, self.vt, self.d_prefix, self.new_prefix, temperature=w.temperature,
                eps=w.eps, delta=w.delta, seed=w.seed, step=0, dev_status=self.status), 1, None))

    def e2e_input(self, name):
        """A per-step input of the end-to-end leg: copied from pinned host
        memory every step into the tensor held by attribute `name`."""
        self.h2d.append((getattr(self, name).cpu().pin_memory(), name))

    # ---- running ---------------------------------------------------------
    def launches_per_step(self):
        return sum(s[2] for s in self.stages)

    def run(self, events=None):
        for i, (_, fn, _, _) in enumerate(self.stages):
            if events is not None:
                events[i].record()
            fn()
        if events is not None:
            events[-1].record()

    def dynamic_bytes(self):
        """Algorithmic bytes of the stages that depend on the accepted path."""
        L = self.acc_len.cpu().numpy().astype(np.int64)
        esz = 2 if self.tdt == self.torch.bfloat16 else 4
        rows = int((L + 1).sum())
        out = {}
        commit = rows * self.w.hkv * self.w.head_dim * 2 * esz * 2
        if self.fused_accept:
            out["kv_commit"] = commit
        elif self.w.accept == "typical":
            out["accept_commit"] = None
        else:
            out["accept_commit"] = rows * self.logits_bytes_row + commit
        return out, float(L.mean())


def _time_calls(call, steps: int, warmup: int, status=None, what: str = ""):
    """Median CUDA-event time of `call` with an L2 flush before each launch
    (the GPU idles while the host queues the events and the launch)."""
    import torch
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    for _ in range(warmup):
        call()
    times = []
    for _ in range(steps):
        flush.fill_(1.0)
        torch.cuda._sleep(2_000_000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(); call(); e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1) * 1e-3)
    if status is not None and int(status.item()) != 0:
        raise RuntimeError(f"{what}: device status {int(status.item())}")
    return statistics.median(times)


def row_timings(device, hbm: float):
    """The rows built on top of the verify step, timed alone at the
    workloads' shapes: the paged prefix cache (70B shape, 128-key blocks in
    a shuffled pool), a 256-node tree (multi-word ancestor masks), rejection
    with stochastic siblings (8B shape), and the LM head fused with greedy
    acceptance against the LM head plus acceptance (Vicuna shape)."""
    import torch
    from tree_speculative_decoding_attn_gb300 import specverify as sv
    from tree_speculative_decoding_attn_gb300 import synth
    out = {}
    r = attention_only("llama70b_serving", device, steps=10, warmup=3, paged=True)
    r["frac_hbm"] = r["gbps"] / hbm
    out["paged_attention_llama70b"] = r
    r = attention_only("long_context", device, steps=10, warmup=3, n_nodes=256, prefix=4096)
    r["frac_hbm"] = r["gbps"] / hbm
    out["attention_256_nodes"] = r
    # stochastic-sibling rejection, 8B shape: batch 8, 60 nodes, vocabulary 128256
    w = synth.WORKLOADS["llama8b_eagle2"]
    B, N, V = w.batch, w.n_nodes, w.vocab
    shape = synth.random_tree(w.seed, N, (10, 4, 3, 2, 2))
    gen = torch.Generator(device=device).manual_seed(w.seed + 5)
    lg = (torch.randn(B, N, V, generator=gen, device=device) * 2).to(torch.bfloat16)
    dq = (torch.randn(B, N, V, generator=gen, device=device) * 2).to(torch.bfloat16)
    i32 = lambda *sh: torch.zeros(sh, dtype=torch.int32, device=device)
    tok, fc, ns = i32(B, N), i32(B, N), i32(B, N)
    cand = torch.from_numpy(synth.candidate_tokens(w.seed, B, shape.n_levels, 10, V)).to(device)
    sv.spec_build_tree(torch.from_numpy(shape.parents).to(device), torch.from_numpy(shape.rank).to(device), cand,
                       i32(B), i32(B), tok, i32(B, N), i32(B, N), torch.zeros((B, N), dtype=torch.int64, device=device),
                       fc, ns)
    par = torch.from_numpy(np.broadcast_to(shape.parents, (B, N)).copy()).to(device)
    al, ap, bo, st = i32(B), i32(B, shape.n_levels + 1), i32(B), i32(1)
    t = _time_calls(lambda: sv.spec_accept(sv.REJECT_STOCHASTIC, lg, tok, par, fc, ns, al, ap, bo, temperature=1.0,
                                           seed=11, step=0, dev_status=st, draft_logits=dq), 10, 3, st, "stochastic")
    out["stochastic_reject_llama8b"] = {"us": t * 1e6, "rows_read_per_visit": 2, "vocab": V, "batch": B}
    del lg, dq
    # LM head + greedy acceptance at the Vicuna shape: fused and as two calls
    w = synth.WORKLOADS["vicuna7b_medusa"]
    B, N, V, d = w.batch, w.n_nodes, w.vocab, w.medusa["hidden"]
    shape = synth.tree_shape(w)
    hid = (torch.randn(B, N, d, generator=gen, device=device)).to(torch.bfloat16)
    wlm = (torch.randn(V, d, generator=gen, device=device) * 0.02).to(torch.bfloat16)
    tok = torch.randint(0, V, (B, N), generator=gen, device=device, dtype=torch.int32)
    fc, ns = i32(B, N), i32(B, N)
    sv.spec_build_tree(torch.from_numpy(shape.parents).to(device), torch.from_numpy(shape.rank).to(device), None,
                       None, i32(B), None, i32(B, N), i32(B, N), torch.zeros((B, N), dtype=torch.int64, device=device),
                       fc, ns)
    par = torch.from_numpy(np.broadcast_to(shape.parents, (B, N)).copy()).to(device)
    al, ap, bo, st = i32(B), i32(B, shape.n_levels + 1), i32(B), i32(1)
    logits = torch.empty(B * N, V, dtype=torch.float32, device=device)
    ws_f = torch.empty(sv.spec_lm_head_accept_workspace_bytes(B, N, d, V), dtype=torch.uint8, device=device)
    ws_l = torch.empty(max(sv.spec_lm_head_workspace_bytes(B * N, d, V), 16), dtype=torch.uint8, device=device)
    t_f = _time_calls(lambda: sv.spec_lm_head_accept(sv.GREEDY, hid, wlm, tok, par, fc, ns, al, ap, bo, workspace=ws_f,
                                                     dev_status=st), 10, 3, st, "fused")
    t_u = _time_calls(lambda: (sv.spec_lm_head(hid.view(B * N, d), wlm, logits, workspace=ws_l, dev_status=st),
                               sv.spec_accept(sv.GREEDY, logits.view(B, N, V), tok, par, fc, ns, al, ap, bo,
                                              dev_status=st)), 10, 3, st, "unfused")
    out["lm_head_accept_vicuna7b"] = {"fused_us": t_f * 1e6, "lm_head_then_accept_us": t_u * 1e6}
    return out


def attention_only(name: str, device, steps: int, warmup: int, paged: bool = False, n_nodes: int = 0,
                   prefix: int = 0):
    """tree_attn_verify alone at a workload's full shape (inputs drawn on the
    device from a seeded torch generator; values do not affect the timing).
    Per-launch CUDA-event times with an L2 flush between launches.  `paged`:
    the prefix cache as 128-key blocks of a shuffled pool; `n_nodes` /
    `prefix`: another tree size (a dense tree) or a uniform prefix length."""
    import torch
    from tree_speculative_decoding_attn_gb300 import specverify as sv
    from tree_speculative_decoding_attn_gb300 import synth
    w = synth.WORKLOADS[name]
    B, N, Hq, Hkv, D = w.batch, n_nodes or w.n_nodes, w.hq, w.hkv, w.head_dim
    prefix = synth.prefix_lengths(w) if not prefix else np.full(B, prefix, np.int32)
    S = int(prefix.max()) + 64
    gen = torch.Generator(device=device).manual_seed(w.seed)
    bf = torch.bfloat16
    rnd = lambda *s: torch.randn(s, generator=gen, device=device, dtype=torch.float32).to(bf)
    q, kt, vt = rnd(B, N, Hq, D), rnd(B, Hkv, N, D), rnd(B, Hkv, N, D)
    blk = 128
    if paged:
        max_blocks = -(-S // blk)
        nb = B * max_blocks
        kc, vc = rnd(nb, Hkv, blk, D), rnd(nb, Hkv, blk, D)
        table = torch.randperm(nb, generator=gen, device=device).to(torch.int32).view(B, max_blocks)
    else:
        kc, vc = rnd(B, Hkv, S, D), rnd(B, Hkv, S, D)
    shape = (synth.dense_tree((8, 4, 4, 2, 2), N) if n_nodes else
             synth.random_tree(w.seed, N, w.caps if w.caps else (10, 4, 3, 2, 2)))
    i32 = lambda *s: torch.zeros(s, dtype=torch.int32, device=device)
    anc = torch.zeros((B, N, sv.mask_words(N)), dtype=torch.int64, device=device).squeeze(-1)
    d_prefix = torch.from_numpy(prefix).to(device)
    sv.spec_build_tree(torch.from_numpy(shape.parents).to(device), torch.from_numpy(shape.rank).to(device), None,
                       None, d_prefix, None, i32(B, N), i32(B, N), anc, i32(B, N), i32(B, N))
    out = torch.empty_like(q)
    splits = sv.tree_attn_plan_splits(bf, B, N, Hq, Hkv, D, prefix)
    wsb = sv.tree_attn_workspace_bytes(bf, B, N, Hq, Hkv, D, int(prefix.max()), splits)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    if paged:
        call = lambda: sv.tree_attn_verify_paged(q, kc, vc, table, kt, vt, d_prefix, anc, out, int(prefix.max()),
                                                 num_splits=splits, workspace=ws, dev_status=status)
    else:
        call = lambda: sv.tree_attn_verify(q, kc, vc, kt, vt, d_prefix, anc, out, int(prefix.max()),
                                           num_splits=splits, workspace=ws, dev_status=status)
    t = _time_calls(call, steps, warmup, status, name)
    nbytes = Hkv * D * 2 * 2 * (int(prefix.sum()) + B * N) + 2 * B * N * Hq * D * 2
    flops = 4 * N * (Hq // Hkv) * D * Hkv * (int(prefix.sum()) + B * N)
    del q, kc, vc, kt, vt
    return {"us": t * 1e6, "gbps": nbytes / t / 1e9, "tflops": flops / t / 1e12, "bytes": nbytes,
            "launches": 2 if wsb else 1, "splits": splits, "n_nodes": N}


# ----------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline leg)
# ----------------------------------------------------------------------------
class OracleStep:
    """One verify step of the CPU oracle on a bounded sample of a workload.

    Inputs are drawn once (untimed); ``step()`` times each stage on its
    sample and extrapolates it to the whole batch by the sampled fraction
    (vocabulary rows/columns for the head and LM-head products, sequences x
    query heads for attention, sequences for acceptance and commit)."""

    def __init__(self, name: str):
        from oracle import tree as T
        from tree_speculative_decoding_attn_gb300 import synth
        self.w = w = synth.WORKLOADS[name]
        B, N, Hq, V = w.batch, w.n_nodes, w.hq, w.vocab
        self.prefix = synth.prefix_lengths(w)
        self.seqs = list(range(min(B, 2)))
        self.heads = list(range(0, Hq, max(1, Hq // 4)))[:4]
        desc = []
        if w.tree == "dynamic":
            dk = w.dynamic
            # (a host-drawn pool of the same shape stands in for the drafting
            # rounds, which the oracle does not time)
            self.pool = synth.candidate_pool(w.seed, B, dk["k"], dk["frontier"], dk["rounds"], V)
            desc.append("drafting rounds not timed (pool drawn)")
        else:
            self.shape = synth.tree_shape(w)
            self.s = w.medusa["topk"] if w.medusa else (max(w.caps) if w.caps else 2)
            self.cand = synth.candidate_tokens(w.seed, B, self.shape.n_levels, self.s, V)
            self.root = synth.root_tokens(w)
        if w.medusa:
            m = w.medusa
            h, w1, w2, wlm = synth.medusa_inputs(w)
            self.rows = np.arange(0, V, max(1, V // 1024))
            self.h, self.w1, self.w2s, self.wlms = h, w1, np.ascontiguousarray(w2[:, self.rows]), \
                np.ascontiguousarray(wlm[self.rows])
            del w2, wlm
            self.head_logits = synth.gaussian(synth.stream(0, "x"), (B * m["heads"], V), 1.0, False)
            self.hid = synth.gaussian(synth.stream(w.seed, "tree_hidden"), (B * N, m["hidden"]), 1.0, True)
            desc.append(f"heads and LM head on {len(self.rows)} of {V} vocabulary rows")
        sub = [int(self.prefix[b]) for b in self.seqs]
        self.att = synth.attention_inputs(w, np.array(sub, np.int32), batch=len(self.seqs))
        self.sub_prefix = np.array(sub, np.int32)
        self.logits = synth.target_logits(w.seed, len(self.seqs), N, V, w.logit_std, w.dtype == "bf16")
        desc.append(f"attention on {len(self.seqs)} of {B} sequences x {len(self.heads)} of {Hq} heads")
        desc.append(f"acceptance and commit on {len(self.seqs)} of {B} sequences")
        self.sample = "; ".join(desc)

    def step(self):
        """Returns (extrapolated seconds for one step, per-stage seconds)."""
        from oracle import accept as ACC
        from oracle import attention as A
        from oracle import commit as COM
        from oracle import heads as H
        from oracle import tree as T
        w = self.w
        B, N, Hq, V = w.batch, w.n_nodes, w.hq, w.vocab
        clock = time.perf_counter
        parts = {}
        if w.tree == "dynamic":
            par, tok, conf = self.pool
            t0 = clock()
            trees = [T.rerank_dynamic(par[b], tok[b], conf[b], N, int(self.prefix[b])) for b in range(B)]
            parts["build_tree"] = clock() - t0
            tree = {k: np.stack([t[k] for t in trees]) for k in ("tok", "parent", "first_child", "next_sibling", "mask")}
        else:
            if w.medusa:
                m = w.medusa
                t0 = clock()
                H.medusa_heads(self.h, self.w1, None, self.w2s)
                t_h = clock() - t0
                frac = (m["hidden"] ** 2 + len(self.rows) * m["hidden"]) / (m["hidden"] ** 2 + V * m["hidden"])
                parts["medusa_heads"] = t_h / frac
                t0 = clock()
                H.topk(self.head_logits, self.s)
                parts["topk"] = clock() - t0
            t0 = clock()
            tree = T.build_tree_static(self.shape.parents, self.shape.rank, self.cand, self.root, self.prefix)
            parts["build_tree"] = clock() - t0
        q, kc, vc, kt, vt = self.att
        t0 = clock()
        for i, b in enumerate(self.seqs):
            A.tree_attention(q[i:i + 1], kc[i:i + 1], vc[i:i + 1], kt[i:i + 1], vt[i:i + 1],
                             self.sub_prefix[i:i + 1], tree["mask"][b], heads=self.heads)
        frac = len(self.seqs) * len(self.heads) * (float(self.sub_prefix.mean()) + N) / \
            (B * Hq * (float(self.prefix.mean()) + N))
        parts["tree_attn"] = (clock() - t0) / frac
        if w.medusa:
            t0 = clock()
            H.lm_head(self.hid, self.wlms)
            parts["lm_head"] = (clock() - t0) * V / len(self.rows)
        sel = {k: tree[k][self.seqs] for k in ("tok", "parent", "first_child", "next_sibling")}
        t0 = clock()
        cap = 8
        if w.accept == "greedy":
            acc = ACC.accept_greedy(self.logits, sel["tok"], sel["first_child"], sel["next_sibling"], cap)
        elif w.accept == "typical":
            acc = ACC.accept_typical(self.logits, sel["tok"], sel["parent"], sel["first_child"], sel["next_sibling"],
                                     w.eps, w.delta, w.temperature, cap)
        else:
            acc = ACC.accept_reject(self.logits, sel["tok"], sel["first_child"], sel["next_sibling"], w.seed, 0,
                                    w.temperature, cap)
        parts["accept"] = (clock() - t0) * B / len(self.seqs)
        t0 = clock()
        COM.kv_commit(kc, vc, kt, vt, self.sub_prefix, acc[0], acc[1])
        parts["kv_commit"] = (clock() - t0) * B / len(self.seqs)
        return sum(parts.values()), parts


def _cpu_baseline_subprocess(name: str, reps: int = 3):
    """Run the oracle timing in a fresh single-threaded process (spawned,
    not forked from this CUDA process)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = (f"import sys, json; sys.path.insert(0, {ROOT!r}); import bench; "
            f"o = bench.OracleStep({name!r}); r = [o.step() for _ in range({reps})]; "
            f"import statistics; print(json.dumps({{'s': statistics.median(x[0] for x in r), 'reps': len(r), "
            f"'sample': o.sample, 'parts': r[0][1]}}))")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    if out.returncode != 0:
        return None, out.stderr[-400:]
    res = json.loads(out.stdout.strip().splitlines()[-1])
    return res, None


# ----------------------------------------------------------------------------
# main
# ----------------------------------------------------------------------------
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        import torch
        rank = int(os.environ.get("RANK", "0"))
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        return dist, rank, local, ws
    return None, 0, 0, 1


def job_max(value: float, dist, device) -> float:
    """Largest per-rank value (seconds) over all ranks; the local value when
    there is a single process."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(steps_per_rank: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: every rank's steps over the slowest rank's time."""
    return world * steps_per_rank / max_seconds


def workload_config(w, world: int) -> dict:
    """The ``config`` object of a bench line (both arms print the same one)."""
    return {"workload": w.name, "batch": w.batch, "hq": w.hq, "hkv": w.hkv, "head_dim": w.head_dim,
            "prefix": list(w.prefix), "n_nodes": w.n_nodes, "vocab": w.vocab, "accept": w.accept,
            "tree": w.tree, "parallelism": f"replicas x{world}",
            "l2": "inputs exceed L2 (weights and/or KV cache streamed each step)"}


def run_reference(args):
    # rank 0 alone times the oracle; other ranks of a torchrun launch exit
    if int(os.environ.get("RANK", "0")) != 0:
        return
    from tree_speculative_decoding_attn_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    o = OracleStep(args.workload)
    for _ in range(min(args.warmup, 1)):  # the oracle has nothing to warm beyond one pass
        o.step()
    # each step runs the oracle on the same bounded sample of the workload;
    # the timed steps stop at a bounded budget of CPU time (the line says how
    # many ran)
    budget_s, spent, measured, extrap = 150.0, 0.0, [], []
    while len(measured) < args.steps and (not measured or spent < budget_s):
        t0 = time.perf_counter()
        s, _ = o.step()
        dt = time.perf_counter() - t0
        spent += dt
        measured.append(dt)
        extrap.append(s)
    sample = f"{o.sample}; {len(measured)} of {args.steps} steps timed (identical deterministic steps)"
    t_full = statistics.median(extrap)
    val = 1.0 / t_full
    line = {"impl": "reference", "metric": "tree-verify steps/s", "value": val, "unit": "steps/s",
            "n_gpus": args.gpus, "steps": len(measured), "warmup": args.warmup,
            # wall time of one sampled oracle step (what the timed region ran)
            "ms_per_step": statistics.median(measured) * 1e3,
            # one whole-workload step, extrapolated from the sample; value = 1 / this
            "ms_per_step_extrapolated": t_full * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, 1),
            "cpu_baseline": {"value": val, "unit": "steps/s", "cores": 1, "kind": "oracle",
                             "sample": sample + " (value extrapolated from the sample by the sampled fraction "
                                                "of each stage)"},
            "e2e": {"value": val, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def capture(step, steps: int, with_events: bool):
    """CUDA graph of ``steps`` verify steps (optionally with a CUDA event
    before every stage, as external record nodes); returns (graph, events)."""
    import torch
    n_st = len(step.stages)
    evs = None
    if with_events:
        mk_ev = lambda: torch.cuda.Event(enable_timing=True, external=True)
        evs = [[mk_ev() for _ in range(n_st + 1)] for _ in range(steps)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for k in range(steps):
            step.run(evs[k] if evs else None)
    torch.cuda.synchronize()
    return graph, evs


def replay_median(graph, min_seconds: float, min_replays: int = 5):
    """Replays ``graph`` back to back for at least ``min_seconds``; returns
    (median replay seconds, replays, wall seconds).  Each replay is timed by
    CUDA events on the current stream."""
    import torch
    times, t_wall = [], time.perf_counter()
    pend = []
    while len(times) + len(pend) < min_replays or time.perf_counter() - t_wall < min_seconds:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(); graph.replay(); e1.record()
        pend.append((e0, e1))
        if len(pend) >= 8:  # bound the queue; keeps the GPU busy back to back
            pend[0][1].synchronize()
            a, b = pend.pop(0)
            times.append(a.elapsed_time(b) * 1e-3)
    torch.cuda.synchronize()
    times += [a.elapsed_time(b) * 1e-3 for a, b in pend]
    return statistics.median(times), len(times), time.perf_counter() - t_wall


def measure_workload(name: str, dev, steps: int, warmup: int, min_seconds: float):
    """Full verify step of one workload: step rate (median graph replay),
    per-stage times (from a second graph with stage events) and the
    attention stage's HBM rate."""
    import torch
    from tree_speculative_decoding_attn_gb300 import specverify as sv
    step = GpuStep(name, dev)
    for _ in range(warmup):
        step.run()
    torch.cuda.synchronize()
    if int(step.status.item()) != 0:
        raise RuntimeError(f"{name}: device status {sv.spec_status_string(int(step.status.item()))}")
    graph, _ = capture(step, steps, False)
    t_rep, reps, _ = replay_median(graph, min_seconds)
    sgraph, evs = capture(step, steps, True)
    sgraph.replay()
    torch.cuda.synchronize()
    n_st = len(step.stages)
    stage_s = {step.stages[i][0]: sum(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(steps)) * 1e-3 / steps
               for i in range(n_st)}
    del graph, sgraph
    res = {"steps_per_s": steps / t_rep, "ms_per_step": t_rep / steps * 1e3, "replays": reps,
           "stages_us": {k: v * 1e6 for k, v in stage_s.items()}, "gpu_launches_per_step": step.launches_per_step()}
    if "tree_attn" in stage_s:
        res["attention_gbps"] = step.attn_bytes / stage_s["tree_attn"] / 1e9
    return step, res, stage_s, t_rep


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=DEFAULT)
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="replay the captured K-step graph back to back for at least this long")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads' step rates and the attention-only timings")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling cases)")
    ap.add_argument("--attention-only", action="store_true",
                    help="time tree_attn_verify alone at the workload's shape (profiling runs)")
    ap.add_argument("--nodes", type=int, default=0,
                    help="with --attention-only: a dense tree of this many nodes instead of the workload's")
    ap.add_argument("--prefix", type=int, default=0,
                    help="with --attention-only: this prefix length for every sequence")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)

    dist, rank, local, ws = _dist()
    import torch
    from tree_speculative_decoding_attn_gb300 import specverify as sv
    from tree_speculative_decoding_attn_gb300 import synth
    sv.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.batch:
        import dataclasses
        synth.WORKLOADS[args.workload] = dataclasses.replace(synth.WORKLOADS[args.workload], batch=args.batch)
    hbm, tc_peak, peak_kind = _peaks()
    if args.attention_only:
        r = attention_only(args.workload, dev, steps=args.steps, warmup=args.warmup, n_nodes=args.nodes,
                           prefix=args.prefix)
        r.update(workload=args.workload, frac_hbm=r["gbps"] / hbm, peak_kind=peak_kind)
        print(json.dumps({"attention_only": r}), flush=True)
        return
    w = synth.WORKLOADS[args.workload]

    # timed region: the K-step graph replayed for >= min_seconds, barrier and
    # synchronize on both sides, clocks sampled throughout
    step = GpuStep(args.workload, dev)
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0, sv.spec_status_string(int(step.status.item()))
    graph, _ = capture(step, args.steps, False)
    graph.replay()  # one untimed replay
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_rep, reps, t_wall = replay_median(graph, args.min_seconds)
    if dist:
        dist.barrier()
    assert int(step.status.item()) == 0, sv.spec_status_string(int(step.status.item()))
    t_rep = job_max(t_rep, dist, dev)
    steps_per_s = job_rate(args.steps, ws, t_rep)
    del graph

    # per-stage times: a second graph of the same K steps with a CUDA event
    # before every stage (the events cost a little; the headline above has none)
    sgraph, evs = capture(step, args.steps, True)
    sgraph.replay()
    torch.cuda.synchronize()
    n_st = len(step.stages)
    stage_s = {step.stages[i][0]: sum(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(args.steps))
               * 1e-3 / args.steps for i in range(n_st)}
    del sgraph
    dyn, mean_acc = step.dynamic_bytes()

    # roofline for the dominant stage
    dom = max(stage_s, key=stage_s.get)
    dom_bytes = next(s[3] for s in step.stages if s[0] == dom)
    if dom_bytes is None:
        dom_bytes = dyn.get(dom)
    roof = None
    if dom_bytes:
        ach = dom_bytes / stage_s[dom] / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "traffic": measured_traffic(args.workload, dom), "peak_kind": peak_kind,
                "bytes_per_launch": dom_bytes, "launch_us": stage_s[dom] * 1e6}

    # end-to-end leg through the public API: every step copies its inputs
    # from pinned host memory and reads its results back.  Two alternating
    # device buffer sets (inputs and results): the input copies run on a
    # stream of their own, so step k + 1's inputs travel while step k
    # computes, and the result read-back on a third, so the next step starts
    # without waiting for it (a set is rewritten only after the step that
    # read its inputs has finished and its results have been read back).
    names = [n for _, n in step.h2d]
    hosts = [h for h, _ in step.h2d]
    h2d_bytes = sum(h.numel() * h.element_size() for h in hosts)
    sets = [[getattr(step, n) for n in names], [torch.empty_like(getattr(step, n)) for n in names]]
    onames = step.d2h_names
    osets = [[getattr(step, n) for n in onames], [torch.empty_like(getattr(step, n)) for n in onames]]
    outs_host = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in osets[0]] for _ in range(2)]
    d2h_bytes = sum(t.numel() * t.element_size() for t in outs_host[0])
    main, copy_s, back_s = torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    freed = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    read = [torch.cuda.Event(), torch.cuda.Event()]

    def use_set(si):
        for n, d in zip(names, sets[si]):
            setattr(step, n, d)
        for n, d in zip(onames, osets[si]):
            setattr(step, n, d)

    def issue_copy(k):
        with torch.cuda.stream(copy_s):
            if k >= 2:
                copy_s.wait_event(freed[k % 2])
            for h, d in zip(hosts, sets[k % 2]):
                d.copy_(h, non_blocking=True)
            copied[k % 2].record(copy_s)

    # each step's API calls once eagerly from Python, and once replayed from
    # a one-step CUDA graph per buffer set (what a serving loop would do);
    # the line reports the graph figure and keeps the eager one beside it
    graphs = []
    for si in range(2):
        use_set(si)
        graphs.append(capture(step, 1, False)[0])

    def e2e_run(use_graphs):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        copy_s.wait_event(e0)
        issue_copy(0)
        for k in range(args.steps):
            if k + 1 < args.steps:
                issue_copy(k + 1)
            main.wait_event(copied[k % 2])
            if k >= 2:
                main.wait_event(read[k % 2])  # this set's previous results are back on the host
            if use_graphs:
                graphs[k % 2].replay()
            else:
                use_set(k % 2)
                step.run()
            freed[k % 2].record(main)
            done[k % 2].record(main)
            with torch.cuda.stream(back_s):
                back_s.wait_event(done[k % 2])
                for hdst, dsrc in zip(outs_host[k % 2], osets[k % 2]):
                    hdst.copy_(dsrc, non_blocking=True)
                read[k % 2].record(back_s)
        main.wait_stream(copy_s)
        main.wait_stream(back_s)
        e1.record()
        torch.cuda.synchronize()
        return job_max(e0.elapsed_time(e1) * 1e-3, dist, dev)

    e2e_eager_s = e2e_run(False)
    e2e_s = e2e_run(True)
    use_set(0)
    del graphs
    e2e = {"value": job_rate(args.steps, ws, e2e_s), "unit": "steps/s", "h2d_bytes_per_step": h2d_bytes,
           "d2h_bytes_per_step": d2h_bytes,
           "how": "per step: H2D of its inputs from pinned memory on a copy stream (double-buffered, "
                  "overlapping the previous step), the step's API calls replayed from a one-step CUDA graph, "
                  "D2H of the accepted paths on a third stream (double-buffered results)",
           "eager_value": job_rate(args.steps, ws, e2e_eager_s)}

    launches = step.launches_per_step()
    attn_s = stage_s.get("tree_attn")
    attention = {"workload": args.workload, "us": attn_s * 1e6, "gbps": step.attn_bytes / attn_s / 1e9,
                 "frac_hbm": step.attn_bytes / attn_s / 1e9 / hbm, "bytes": step.attn_bytes}
    del step
    torch.cuda.empty_cache()

    extra, extra_attn, rows = {}, {}, {}
    if rank == 0 and not args.no_extra:
        for nm in synth.WORKLOADS:
            if nm == args.workload:
                continue
            st, res, _, _ = measure_workload(nm, dev, args.steps, 3, min_seconds=0.2)
            if "attention_gbps" in res:
                res["attention_frac_hbm"] = res["attention_gbps"] / hbm
            extra[nm] = res
            del st
            torch.cuda.empty_cache()
        for nm in ("llama8b_eagle2", "llama70b_serving", "long_context"):
            r = attention_only(nm, dev, steps=20, warmup=3)
            r["frac_hbm"] = r["gbps"] / hbm
            r["frac_tensor"] = r["tflops"] / tc_peak
            extra_attn[nm] = r
            torch.cuda.empty_cache()
        rows = row_timings(dev, hbm)
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        res, err = _cpu_baseline_subprocess(args.workload)
        if res:
            cpu = {"value": 1.0 / res["s"], "unit": "steps/s", "cores": 1, "kind": "oracle",
                   "sample": res["sample"] + f" (median of {res['reps']} steps, each extrapolated by the sampled "
                                             "fraction of each stage)"}
        else:
            cpu = {"value": None, "unit": "steps/s", "cores": 1, "kind": "oracle", "sample": f"failed: {err}"}

    if rank == 0:
        line = {"metric": "tree-verify steps/s", "value": steps_per_s, "unit": "steps/s", "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_rep / args.steps * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic (seeded; random weights)",
                "config": workload_config(w, ws),
                "timing": {"launch": "cuda_graph", "replays": reps, "replay_s_median": t_rep, "timed_wall_s": t_wall,
                           "how": "median CUDA-event time of back-to-back replays of one K-step graph"},
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches * args.steps,
                "stages_us": {k: v * 1e6 for k, v in stage_s.items()},
                "mean_accepted": mean_acc, "attention": attention, "workloads": extra,
                "attention_full_shapes": extra_attn, "rows": rows, "clocks": clocks.summary()}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
