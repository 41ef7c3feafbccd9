"""Benchmark of the Token Recycling per-step hot path on one GB300 (or N, weak scaling).

A step is one pass of the whole hot path over one batch: tree-attention
verification (tr_verify_attn), then tr_step (top-K or fused LM head + top-K,
greedy acceptance, matrix update, KV commit, next tree retrieval).  The
synthetic target that produces each step's logits depends on that step's
tree, so the timed run replays a recording: the loop first runs with the
device-side target, storing every step's logits (or hidden states) and
attention operands in HBM; the state is then restored and the same steps run
again with only the hot-path kernels inside the timed region.  The replay must
end in the recorded state, which is checked.  Inputs of every step are larger
than L2 (fresh logits and the KV cache), so no flush is needed between steps.

Default workload: 16 sequences with their own matrices (V=32000, K=8, int64),
80-node tree, prefixes uniform in 1k..4k, 32 heads x 128, fp32 logits.

--impl reference times the CPU oracle (a deliberately plain program) on a
bounded sample of the same workload instead.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

PEAK_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# dram bytes per launch of the dominant kernel from an ncu capture of this
# workload (dram__bytes_read.sum + dram__bytes_write.sum, mean of three launches),
# valid only while the kernel's sources are unchanged (sha256 of the files)
TRAFFIC = {"attn": {"bytes": 631514000 + 2531000, "sha": "e0ee697942013f87", "files": ("tr_attn.cu", "tr_sm100.cuh")}}


PRIME_CYCLES = 2_000_000   # about 1 ms of device time at the GB300's clocks

# ex2.approx.f32 results per SM per clock on this GPU, measured with a loop of
# independent exponentials at 4, 8 and 16 warps per SM (31.7 - 32.8)
EXP2_PER_SM_CLK = 32


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAK_FALLBACK, "fallback"


U_SEED = 0xACC_E97   # seed of the acceptance uniforms under sampling
INIT_SEED = 0x5EED_0F_7E57


def config_of(args, wl, world):
    """The workload as both arms name it in their JSON line."""
    return {"workload": args.workload, "B": wl.B, "V": wl.V, "K": wl.K, "tree": wl.tree, "tree_nodes": wl.N,
            "tree_depth": wl.depth(), "prefix": list(wl.prefix), "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
            "acceptance": ("greedy" if args.temperature is None else "sampled at T=%g" % args.temperature),
            "init": args.init, "update": args.update,
            **({"lm_operands": args.lm_operands} if wl.logits == "lmhead" else {}),
            "parallelism": "replicas (dp%d, no collective)" % world,
            "l2": ("every step reads its own recorded hidden rows; the weight (V x D bf16) is larger than L2"
                   if wl.logits == "lmhead" else
                   "every step reads its own recorded logits and Q/K/V (all steps together far larger than L2) "
                   "and the KV cache")}


def src_sha(*names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "free_speculative_decoding_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def attn_bytes(w, N, L):
    """Algorithmic HBM bytes of one tr_verify_attn launch with cache lengths L[b]:
    cached K and V read once, tree Q/K/V read once, fp32 O written once."""
    kv = 2 * 2 * w.Hkv * w.d * int(np.sum(L))
    tree = w.B * N * w.d * 2 * (w.Hq + 2 * w.Hkv)
    out = w.B * N * w.Hq * w.d * 4
    return kv + tree + out


def attn_flops(w, N, L):
    """Algorithmic tensor work of one tr_verify_attn launch: Q.K^T and P.V over
    every key a node's tile holds (the L_b cached keys and the N tree rows),
    2 flops per multiply-add; the exponentials: one per (query head, node, key)."""
    keys = int(np.sum(np.asarray(L, dtype=np.int64) + N))
    return 4.0 * w.Hq * N * w.d * keys, float(w.Hq * N * keys)


def launches_per_step(w):
    """libtr kernels launched by one timed step: verify attention (1), then
    tr_step = top-K (1) or fused LM head (tile + merge, 2), and the fused
    accept/update/commit/retrieve kernel (1)."""
    return (1 if w.attention else 0) + (2 if w.logits == "lmhead" else 1) + 1


def topk_bytes(w, N):
    esz = 2 if w.logits == "bf16" else 4
    return w.B * N * w.V * esz


def workload_of(args):
    """The named workload, with the draft tree of --tree if given."""
    w = synth.WORKLOADS[args.workload]
    return w.scaled(tree=args.tree) if args.tree else w


def rank_workload(w, rank, world):
    """The workload of one rank: each rank decodes its own sequences (the seed
    moves with the rank); shapes are the same on every rank."""
    return w.scaled(seed=w.seed + 1000 * rank) if world > 1 else w


def max_over_ranks(x, world, device):
    """The largest of the ranks' values (the job's time is its slowest rank)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, steps, total_ms):
    """Whole-job steps/s: every rank ran `steps` steps of its own batch within total_ms."""
    return world * steps * 1e3 / total_ms


def run_gpu(args, rank, world):
    import torch

    import free_speculative_decoding_gb300 as tr
    from free_speculative_decoding_gb300.engine import TRState
    from synth import device as sd

    w = rank_workload(workload_of(args), rank, world)
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    tree = tr.Tree(w.child_counts, w.K)
    N = tree.N
    mdt = torch.int64 if w.m_dtype == "int64" else torch.int32
    ldt = torch.bfloat16 if w.logits == "bf16" else torch.float32
    lm = w.logits == "lmhead"
    W, K = args.warmup, args.steps
    cap = int(w.prefix[1]) + (W + K) * (tree.max_depth + 1)
    st = TRState(tree, w.B, w.V, m_dtype=mdt, Hq=w.Hq if w.attention else 0, Hkv=w.Hkv, d=w.d, cap=cap,
                 logits_dtype=ldt, D=w.D if lm else 0, device=dev)
    tgt = sd.DeviceTarget(w, tree, dev)
    realistic = lm and args.lm_operands == "realistic"
    if realistic:
        # off-grid operands: the weight ~ N(0, 0.02^2) and every step's hidden
        # rows ~ N(0, 1) in bf16, full mantissas (timing only: such a target
        # does not depend on the tokens, so acceptance is incidental)
        gen = torch.Generator(device=dev).manual_seed(w.seed)
        tgt.Wt.copy_((torch.randn(w.V, w.D, generator=gen, device=dev) * 0.02).to(torch.bfloat16))
    if w.attention:
        sd.fill_cache(w, st)
    start_matrices(args, w, st)
    stream = torch.cuda.current_stream()
    T = args.temperature
    upd = tr.TR_UPD_ACCEPTED if args.update == "accepted" else tr.TR_UPD_ALL

    # per-step input sizes
    if lm:
        step_in = w.B * N * w.D * 2
    else:
        step_in = w.B * N * w.V * (2 if w.logits == "bf16" else 4)
    qkv_b = w.B * N * w.d * 2 * (w.Hq + 2 * w.Hkv) if w.attention else 0
    if T is not None:
        step_in += w.B * N * (w.K + 1) * 4   # the acceptance uniforms
    budget = args.store_gb * 2 ** 30
    seg = max(1, min(K, int(budget // max(1, step_in + qkv_b))))

    def make_bufs(n):
        bufs = {}
        if lm:
            bufs["H"] = torch.empty(n, w.B * N, w.D, dtype=torch.bfloat16, device=dev)
        else:
            bufs["logits"] = torch.empty(n, w.B * N, w.V, dtype=ldt, device=dev)
        if w.attention:
            bufs["q"] = torch.empty(n, w.B, N, w.Hq, w.d, dtype=torch.bfloat16, device=dev)
            bufs["kt"] = torch.empty(n, w.B, N, w.Hkv, w.d, dtype=torch.bfloat16, device=dev)
            bufs["vt"] = torch.empty(n, w.B, N, w.Hkv, w.d, dtype=torch.bfloat16, device=dev)
        if T is not None:
            bufs["U"] = torch.empty(n, w.B, N, w.K + 1, dtype=torch.float32, device=dev)
        return bufs

    bufs = make_bufs(seg)
    gstep = [0]

    def gen_step(i):
        """Generate step inputs into slot i for the current tree (the target stand-in)."""
        s = gstep[0]
        if w.attention:
            sd.step_qkv(w, s, N, dev, out=(bufs["q"][i], bufs["kt"][i], bufs["vt"][i]))
        if realistic:
            bufs["H"][i].copy_(torch.randn(w.B * N, w.D, generator=gen, device=dev).to(torch.bfloat16))
        elif lm:
            tgt.hidden_for(st, bufs["H"][i])
        else:
            tgt.logits_for(st, bufs["logits"][i])
        if T is not None:
            tr.trsyn_uniforms(U_SEED, s, bufs["U"][i])
        gstep[0] += 1

    def hot_step(i, ev=None):
        kt = vt = None
        if ev is not None:
            ev[0].record(stream)
        if w.attention:
            kt, vt = bufs["kt"][i], bufs["vt"][i]
            st.verify(bufs["q"][i], kt, vt)
        if ev is not None:
            ev[1].record(stream)
        if lm:
            st.finish(H=bufs["H"][i], Wt=tgt.Wt, Kt=kt, Vt=vt, mode=upd)
        elif T is not None:
            st.finish(logits=bufs["logits"][i], Kt=kt, Vt=vt, mode=upd, temperature=T, U=bufs["U"][i])
        else:
            st.finish(logits=bufs["logits"][i], Kt=kt, Vt=vt, mode=upd)
        if ev is not None:
            ev[2].record(stream)

    def snapshot():
        snap = {"M": st.M.clone(), "root": st.root.clone(), "L": st.L.clone(), "tok": st.tree_tok.clone()}
        return snap

    def restore(snap):
        st.M.copy_(snap["M"])
        st.root.copy_(snap["root"])
        st.L.copy_(snap["L"])
        st.tree_tok.copy_(snap["tok"])

    # warm-up: W full steps (target + hot path), untimed
    for _ in range(W):
        gen_step(0)
        hot_step(0)
    torch.cuda.synchronize()

    if world > 1:
        import torch.distributed as dist
        dist.barrier()

    total_ms = 0.0
    attn_ms, step_ms = [], []
    attn_bytes_list = []
    attn_work = []
    done = 0
    replay_ok = True
    committed = 0
    clocks = ClockSampler(dev.index)
    clocks_started = False
    while done < K:
        n = min(seg, K - done)
        snap = snapshot()
        L_hist = []
        # record: the target writes each step's inputs for the tree of that step
        for i in range(n):
            L_hist.append(st.L.clone())
            gen_step(i)
            hot_step(i)
        ref_state = (st.M.clone(), st.L.clone(), st.root.clone())
        restore(snap)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if not clocks_started:
            clocks.start()
            clocks_started = True
            time.sleep(0.3)
        torch.cuda.synchronize()
        # a short device-side spin ahead of the start event lets the host queue
        # the first launches before the clock starts, so the timed region holds
        # device work only (the e2e line below keeps the host path)
        torch.cuda._sleep(PRIME_CYCLES)
        start.record(stream)
        for i in range(n):
            hot_step(i, evs[i])
        stop.record(stream)
        torch.cuda.synchronize()
        total_ms += start.elapsed_time(stop)
        for i in range(n):
            if w.attention:
                attn_ms.append(evs[i][0].elapsed_time(evs[i][1]))
                attn_bytes_list.append(attn_bytes(w, N, L_hist[i].cpu().numpy()))
                attn_work.append(attn_flops(w, N, L_hist[i].cpu().numpy()))
            step_ms.append(evs[i][1].elapsed_time(evs[i][2]))
        replay_ok &= bool(torch.equal(st.M, ref_state[0]) and torch.equal(st.L, ref_state[1])
                          and torch.equal(st.root, ref_state[2]))
        committed += int((st.L - snap["L"]).sum().item())
        done += n
    clk = clocks.stop()
    status = st.status()

    # tr_topk alone on the recorded logits (outside the timed region): each
    # launch reads another step's logits, so the input is not in L2
    topk_ms = []
    if not lm:
        nslot = min(seg, K)
        rows = w.B * N
        ids = torch.empty(rows, w.K, dtype=torch.int32, device=dev)
        vals = torch.empty(rows, w.K, dtype=torch.float32, device=dev)
        ws = tr.workspace(tr.tr_topk_workspace_bytes(rows, w.V, w.K), dev)
        if nslot >= 2:
            for j in range(3):
                tr.tr_topk(bufs["logits"][j % nslot], w.K, ids, vals, ws)
            tev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(max(8, nslot))]
            torch.cuda.synchronize()
            # the same device-side spin: every launch is queued before the
            # first start event, so each interval holds the kernel alone
            torch.cuda._sleep(2 * PRIME_CYCLES)
            for j, (e0, e1) in enumerate(tev):
                e0.record(stream)
                tr.tr_topk(bufs["logits"][j % nslot], w.K, ids, vals, ws)
                e1.record(stream)
            torch.cuda.synchronize()
            topk_ms = [e0.elapsed_time(e1) for e0, e1 in tev]

    total_ms = max_over_ranks(total_ms, world, dev)

    res = {"total_ms": total_ms, "attn_ms": attn_ms, "attn_bytes": attn_bytes_list, "attn_work": attn_work,
           "sm_count": torch.cuda.get_device_properties(dev).multi_processor_count, "replay_ok": replay_ok,
           "status": status, "clocks": clk, "committed": committed, "N": N, "w": w, "seg": seg,
           "step_ms": step_ms, "topk_ms": topk_ms}

    # end to end through the public calls with host buffers (rank 0 and every rank alike)
    if args.e2e_steps > 0:
        res["e2e"] = run_e2e(args, w, st, tgt, bufs, gen_step, hot_step, snapshot, restore, dev, N, lm)
    return res


def start_matrices(args, w, st):
    """Initial matrices and first trees: the workload's synthetic inherited
    matrices (each sequence inherits its own through tr_init_matrix), or an
    all-zero / random start (tr_init_matrix over the batch)."""
    import free_speculative_decoding_gb300 as tr
    from synth import device as sd
    roots, L0 = synth.initial_roots(w), w.prefix_lengths()
    if args.init == "inherit":
        sd.warm_matrices(w, st)
        src = st.M.clone()
        for b in range(w.B):
            tr.tr_init_matrix(st.M[b:b + 1], tr.TR_INIT_INHERIT, src[b])
        st.start(roots, L0, M_src=None, mode=None)
    else:
        st.start(roots, L0, M_src=None, mode=tr.TR_INIT_ZERO if args.init == "zero" else tr.TR_INIT_RANDOM,
                 seed=INIT_SEED)


def run_e2e(args, w, st, tgt, bufs, gen_step, hot_step, snapshot, restore, dev, N, lm):
    """Same steps with every step's inputs copied from pinned host memory and the
    committed tokens read back, all inside the timed region.  The copy of step
    i+1's inputs overlaps step i on a second stream (two device slots)."""
    import torch

    E = min(args.e2e_steps, bufs["H" if lm else "logits"].shape[0])
    snap = snapshot()
    for i in range(E):
        gen_step(i)
        hot_step(i)
    restore(snap)
    torch.cuda.synchronize()
    host = {k: torch.empty(v[:E].shape, dtype=v.dtype, pin_memory=True) for k, v in bufs.items()}
    for k in host:
        host[k].copy_(bufs[k][:E])
    out_acc = torch.empty(E, w.B, dtype=torch.int32, pin_memory=True)
    out_com = torch.empty(E, w.B, st.committed.shape[1], dtype=torch.int32, pin_memory=True)
    h2d = sum(host[k][0].numel() * host[k][0].element_size() for k in host)
    d2h = out_acc[0].numel() * 4 + out_com[0].numel() * 4
    stream = torch.cuda.current_stream()
    # two device slots: a copy stream brings step i+1's inputs in while step i
    # runs; slot reuse waits for the step that last read it (splitting the
    # copy over several streams measured no faster)
    copy_stream = torch.cuda.Stream(device=dev)
    slots = 2 if bufs["H" if lm else "logits"].shape[0] >= 2 else 1
    copied = [torch.cuda.Event() for _ in range(E)]
    used = [torch.cuda.Event() for _ in range(E)]

    def copy_in(i):
        with torch.cuda.stream(copy_stream):
            if i >= slots:
                copy_stream.wait_event(used[i - slots])
            for k in host:
                bufs[k][i % slots].copy_(host[k][i], non_blocking=True)
            copied[i].record(copy_stream)

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    copy_stream.wait_event(start)
    copy_in(0)
    for i in range(E):
        if i + 1 < E:
            copy_in(i + 1)
        stream.wait_event(copied[i])
        hot_step(i % slots)
        used[i].record(stream)
        out_acc[i].copy_(st.acc_len, non_blocking=True)
        out_com[i].copy_(st.committed, non_blocking=True)
    stop.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms = start.elapsed_time(stop)
    restore(snap)
    return {"steps": E, "ms": ms, "wall_s": wall, "h2d": int(h2d), "d2h": int(d2h)}


# ----------------------------------------------------------------------------
# oracle arm (CPU)
# ----------------------------------------------------------------------------

def oracle_sequence_step(w, b, state, plan, step, temperature=None, mode=0):
    """One Token Recycling step of sequence b on the CPU oracle; returns seconds
    spent in the method (the synthetic target's logits are made before timing)."""
    import oracle
    depth = np.asarray(plan.depth)
    U = synth.uniforms(U_SEED, step, b, plan.N, w.K + 1) if temperature is not None else None
    tok = oracle.retrieve(state.M, state.root, plan)
    if w.logits == "lmhead":
        H = synth.bf16_to_f32(synth.lm_hidden_rows(w.seed, b, state.L + depth, tok, w.D))
        Wt = _lm_weight_cache(w)
        t0 = time.perf_counter()
        tok = oracle.retrieve(state.M, state.root, plan)
        rows = oracle.lmhead_logits(H, Wt)
    else:
        rows = synth.logits_f32(w.seed, b, state.L + depth, tok, w.V, w.logits)
        qkv = None
        if w.attention:
            q, kt, vt = synth.step_qkv(w, step, [b])
            qkv = (synth.bf16_to_f32(q[0]), synth.bf16_to_f32(kt[0]), synth.bf16_to_f32(vt[0]))
        t0 = time.perf_counter()
        tok = oracle.retrieve(state.M, state.root, plan)
        if qkv is not None:
            oracle.tree_attention(qkv[0], state.kc, state.vc, state.L, qkv[1], qkv[2], plan, w.d ** -0.5)
    ids, _ = oracle.topk_rows(rows, w.K)
    if temperature is None:
        acc, path, committed, bonus = oracle.accept(plan, tok, ids[:, 0])
    else:
        acc, path, committed, bonus, _, _ = oracle.accept_sampled(plan, tok, rows, temperature, U)
    oracle.update(state.M, tok, ids, plan, mode, path)
    if w.attention and state.kc is not None:
        state.L = oracle.kv_commit(state.kc, state.vc, qkv[1], qkv[2], state.L, path)
    else:
        state.L += len(path)
    state.root = bonus
    return time.perf_counter() - t0


_LMW = {}


def _lm_weight_cache(w):
    if w.name not in _LMW:
        _LMW[w.name] = synth.bf16_to_f32(synth.lm_weight_rows(w.seed, w.V, w.D)).astype(np.float64)
    return _LMW[w.name]


def oracle_matrix(w, b, init):
    import oracle
    if init == "zero":
        return oracle.init_matrix(oracle.INIT_ZERO, w.V, w.K)
    if init == "random":
        return oracle.init_matrix(oracle.INIT_RANDOM, w.V, w.K, seed=INIT_SEED, seq=b)
    return synth.warm_matrix(w.seed, b, w.V, w.K)


def oracle_rate(w, budget_s, max_seq_steps=None, temperature=None, init="inherit", update="all"):
    """Oracle steps/s of the full batch, extrapolated from a bounded sample of
    sequence-steps of one sequence (each sequence is independent and alike)."""
    import oracle
    plan = oracle.TreePlan(w.child_counts, w.K)
    b = 0
    L0 = int(w.prefix_lengths()[b])
    mode = oracle.UPD_ACCEPTED if update == "accepted" else oracle.UPD_ALL
    st = oracle.TRState(M=oracle_matrix(w, b, init), root=int(synth.initial_roots(w)[b]), L=L0)
    if w.attention:
        cap = L0 + 64 * (plan.max_depth + 1)
        st.kc = np.zeros((w.Hkv, cap, w.d), np.float32)
        st.vc = np.zeros_like(st.kc)
        hh, pp = np.meshgrid(np.arange(w.Hkv), np.arange(L0), indexing="ij")
        st.kc[:, :L0] = synth.bf16_to_f32(synth.kc_rows(w.seed, b, hh, pp, w.d)).reshape(w.Hkv, L0, w.d)
        st.vc[:, :L0] = synth.bf16_to_f32(synth.vc_rows(w.seed, b, hh, pp, w.d)).reshape(w.Hkv, L0, w.d)
    spent, n = 0.0, 0
    while spent < budget_s and (max_seq_steps is None or n < max_seq_steps) and n < 64:
        spent += oracle_sequence_step(w, b, st, plan, n, temperature, mode)
        n += 1
    per_seq_step = spent / n
    return 1.0 / (per_seq_step * w.B), n, spent


def cpu_cores():
    """The host cores this process may run on (numpy's BLAS may use them all)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_rate_one_core(args, budget_s, max_seq_steps=None):
    """oracle_rate on one core: a child process pinned to one CPU with one BLAS
    thread.  Returns a cpu_baseline-style dict, or None if the child failed."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               RANK="0", WORLD_SIZE="1")
    code = ("import os, sys, json, types\n"
            "os.sched_setaffinity(0, {min(os.sched_getaffinity(0))})\n"
            "sys.path.insert(0, %r)\n"
            "import bench\n"
            "w = bench.workload_of(types.SimpleNamespace(workload=%r, tree=%r))\n"
            "print(json.dumps(bench.oracle_rate(w, %r, %r, %r, %r, %r)))\n"
            % (ROOT, args.workload, args.tree, float(budget_s), max_seq_steps, args.temperature, args.init,
               args.update))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
        rate, n, spent = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception:
        return None
    return {"value": rate, "cores": 1,
            "sample": "%d sequence-steps of sequence 0 (%.1f s) on one pinned core, one BLAS thread" % (n, spent)}


# ----------------------------------------------------------------------------
# main
# ----------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", default="tr", choices=["tr", "reference"])
    ap.add_argument("--workload", default="batched", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--tree", default=None, choices=sorted(synth.TREES),
                    help="draft tree in place of the workload's own (the tree-shape sweep)")
    ap.add_argument("--store-gb", type=float, default=40.0, help="HBM for recorded step inputs")
    ap.add_argument("--e2e-steps", type=int, default=16)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--temperature", type=float, default=None,
                    help="acceptance under sampling at this temperature (tr_step_sampled); greedy without it")
    ap.add_argument("--init", default="inherit", choices=["inherit", "zero", "random"],
                    help="starting matrices: each sequence's inherited synthetic matrix, all zero, or random")
    ap.add_argument("--update", default="all", choices=["all", "accepted"],
                    help="matrix update from every verified node, or from the accepted path only")
    ap.add_argument("--lm-operands", default="grid", choices=["grid", "realistic"],
                    help="fused LM-head workload: the grid-valued synthetic target, or off-grid N(0,1) hidden "
                         "rows and N(0, 0.02^2) weights (timing only)")
    args = ap.parse_args()
    if args.temperature is not None and synth.WORKLOADS[args.workload].logits == "lmhead":
        ap.error("sampling needs stored logits: not with the fused LM-head workload")

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    w = workload_of(args)
    metric = "TR steps/s"
    unit = "steps/s (%d sequences x %d-node tree per step)" % (w.B, w.N)

    if args.impl == "reference":
        if rank != 0:
            return
        per_step = max(1.0, 150.0 / max(1, args.steps + args.warmup))
        import oracle  # noqa: F401
        okw = dict(temperature=args.temperature, init=args.init, update=args.update)
        oracle_rate(w, budget_s=1e9, max_seq_steps=max(1, args.warmup), **okw)   # warm-up steps
        rate, n, spent = oracle_rate(w, budget_s=per_step * args.steps, max_seq_steps=args.steps, **okw)
        line = {"impl": "reference", "metric": metric, "value": rate, "unit": unit, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / rate, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64 attention / exact compare", "data": "synthetic",
                "config": config_of(args, w, world), "timed": "the oracle on a bounded sample of the workload",
                "cpu_baseline": {"value": rate, "unit": unit, "cores": cpu_cores(), "kind": "oracle",
                                 "sample": "%d sequence-steps of sequence 0 (%.1f s), scaled to %d sequences"
                                           % (n, spent, w.B)},
                "e2e": {"value": rate, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        if args.workload == "tiny":
            # the latency-bound single-sequence loop: also its one-core oracle rate
            one = oracle_rate_one_core(args, per_step * args.steps, args.steps)
            if one:
                line["cpu_baseline"]["one_core"] = one
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))))
    res = run_gpu(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    K = args.steps
    wl = res["w"]
    N = res["N"]
    ms_per_step = res["total_ms"] / K
    value = job_rate(world, K, res["total_ms"])   # whole-job steps/s (each rank its own batch)
    peaks, peak_kind = load_peaks()
    roofline = None
    if wl.attention and res["attn_ms"]:
        a_ms = float(np.mean(res["attn_ms"]))
        a_bytes = float(np.mean(res["attn_bytes"]))
        ach = a_bytes / (a_ms * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        tr_ = TRAFFIC.get("attn")
        traffic = tr_["bytes"] if tr_ and tr_["sha"] == src_sha(*tr_["files"]) and args.workload == "batched" else None
        flops, exps = (float(np.mean(x)) for x in zip(*res["attn_work"]))
        tf = flops / (a_ms * 1e-3) / 1e12
        # exp2: 32 per SM per clock, measured on this GPU with a loop of
        # independent ex2.approx.ftz.f32 (31.7-32.8 at 4-16 warps per SM)
        sm_mhz = res["clocks"].get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
        exp_peak = EXP2_PER_SM_CLK * res["sm_count"] * sm_mhz * 1e6 / 1e9
        exp_rate = exps / (a_ms * 1e-3) / 1e9
        hbm = {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak}
        tensor = {"bound": "tensor", "achieved": tf, "peak": float(peaks["bf16_tflops"]), "unit": "TFLOP/s",
                  "frac": tf / float(peaks["bf16_tflops"]), "flops_per_launch": flops}
        exp = {"achieved": exp_rate, "peak": exp_peak, "unit": "Gexp2/s", "frac": exp_rate / exp_peak,
               "peak_source": "%d exp2 per SM per clock (measured) x %d SMs x %.0f MHz"
                              % (EXP2_PER_SM_CLK, res["sm_count"], sm_mhz)}
        # grouped-query heads read each K/V tile for several query heads: the
        # tensor pipe, not HBM, is the bound there
        main, other = (tensor, hbm) if wl.Hq != wl.Hkv else (hbm, tensor)
        roofline = dict(kernel="tr_verify_attn", **main, traffic=traffic if main is hbm else None,
                        peak_source=peak_kind + (" bf16 dense (burst)" if main is tensor else ""),
                        algorithmic_bytes_per_launch=a_bytes, ms_per_launch=a_ms,
                        **{"also_" + other["bound"]: other}, exp2=exp)
    if wl.logits == "lmhead" and res["step_ms"]:
        s_ms = float(np.mean(res["step_ms"]))
        flops = 2.0 * wl.B * N * wl.D * wl.V
        ach = flops / (s_ms * 1e-3) / 1e12
        peak = float(peaks["bf16_tflops"])
        roofline = {"kernel": "tr_step (fused LM head + top-K, merge, accept/update)", "bound": "tensor",
                    "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak, "traffic": None,
                    "peak_source": peak_kind + " bf16 dense (burst)", "flops_per_launch": flops,
                    "ms_per_launch": s_ms}
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 attention (fp32 accumulate), %s logits, int64/int32 state" % wl.logits,
        "data": "synthetic: seeded splitmix64 Markov-plus-noise target logits, Irwin-Hall bf16 attention operands",
        "config": config_of(args, wl, world), "timed": "record-then-replay: hot-path kernels only",
        "tree_tokens_per_s": value * wl.B * N,
        "committed_tokens_per_s": world * res["committed"] / (res["total_ms"] * 1e-3),
        "mat": res["committed"] / (K * wl.B),
        "replay_matches_record": res["replay_ok"], "device_status": res["status"],
        "gpu_launches": K * launches_per_step(wl),
        "clocks": res["clocks"],
    }
    if res["step_ms"]:
        line["tr_step_ms"] = float(np.mean(res["step_ms"]))
        line["topk_bytes_per_launch"] = topk_bytes(wl, N)
    if roofline:
        line["roofline"] = roofline
    if res["topk_ms"]:
        t_ms = float(np.mean(res["topk_ms"]))
        t_b = topk_bytes(wl, N)
        line["kernels"] = {"tr_topk": {
            "bound": "hbm", "ms_per_launch": t_ms, "algorithmic_bytes_per_launch": t_b,
            "achieved": t_b / (t_ms * 1e-3) / 1e9, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
            "frac": t_b / (t_ms * 1e-3) / 1e9 / float(peaks["hbm_gbs"]),
            "timed": "alone, after the timed region, over %d recorded steps' logits (each larger than L2)"
                     % len(res["topk_ms"])}}
    if "e2e" in res:
        e = res["e2e"]
        line["e2e"] = {"value": world * e["steps"] / (e["ms"] * 1e-3), "unit": unit, "h2d_bytes_per_step": e["h2d"],
                       "d2h_bytes_per_step": e["d2h"], "steps": e["steps"]}
    # the oracle on a bounded sample of the same workload, on this host's cores
    rate, n, spent = oracle_rate(wl, budget_s=args.cpu_budget, temperature=args.temperature, init=args.init,
                                 update=args.update)
    line["cpu_baseline"] = {"value": rate, "unit": unit, "cores": cpu_cores(), "kind": "oracle",
                            "sample": "%d sequence-steps of sequence 0 (%.1f s of oracle time), scaled to %d "
                                      "sequences; BLAS calls may use all cores" % (n, spent, wl.B)}
    if args.workload == "tiny" and world == 1:
        one = oracle_rate_one_core(args, args.cpu_budget)
        if one:
            line["cpu_baseline"]["one_core"] = one
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
