#!/usr/bin/env python3
"""Benchmark of one speculative cycle: context injection, the single-pass
block draft and verification, on the full drafter dimensions.

A step is one cycle for every request of the batch:
  dflash_ctx_append  (features of the tau positions the target scored last cycle)
  dflash_draft_block (anchor + 7 MASK, 5 layers, LM head, top-4)
  dflash_verify      (greedy; writes the next anchor and append count on device)
The target model is not part of this path: its logits are stood in for by the
draft logits plus N(0, sigma) noise, formed by two torch ops whose time is
measured separately and excluded (latency per token L = (T_draft + T_verify)
/ tau, blog "DFlash vs DFlash 2", section "The problem: one expensive token at
a time").  The whole step is captured once in a CUDA graph and replayed.

The headline line is batch 1, gamma 8 (context 4,096, greedy).  Beside it the
line carries the other workloads of the same metric: batch 16 with
log-uniform contexts and sampled verification, batch 32 at gamma 8 (greedy
and sampled) and at gamma 16, each as a whole cycle with its verified tokens
per second, and a verify-only sweep (batch 1..256 x gamma 8/16 x noise).

Prints one JSON line (rank 0).  --impl reference times the float64 CPU
oracle on the host cores instead (bounded sample per step, scaled).
--gpus N without torchrun starts N replica ranks itself.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "draft blocks/s and verified tokens/s (γ=8) at batch 1/16/32; % HBM/TC roofline"
DIMS_FULL = dict(d=5120, n_q=40, n_kv=8, hd=128, ffn=17408, vocab=151936, n_layers=5,
                 n_feat=5, feat_dim=5120, window=4096)
WORKLOAD = ("full drafter dims (5 layers, hidden 5120, 40q/8kv x 128, SwiGLU 17408, vocab 151936), "
            "batch {B}, gamma {G}, context {L} filling the 4096 window, top-4, greedy verify")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--gamma", type=int, default=8)
    ap.add_argument("--context", type=int, default=4096)
    ap.add_argument("--sigma", type=float, default=0.05,
                    help="std of the noise that turns draft logits into stand-in target logits")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the batch 16/32 lines and the verify sweep")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--profile-cycles", type=int, default=0,
                    help="profiling case: run this many eager cycles and exit (for ncu)")
    ap.add_argument("--layers", type=int, default=5, help="drafter layers (profiling cases only)")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "e4m3"],
                    help="drafter weight format of the profiling case (--profile-cycles)")
    ap.add_argument("--sampled", action="store_true",
                    help="sampled drafting and verification in the profiling case (--profile-cycles)")
    ap.add_argument("--cpu-probe", default=None, choices=["tiny", "verify16"],
                    help=argparse.SUPPRESS)  # one oracle timing, run in a child process
    return ap.parse_args()


def spawn_replicas(args):
    """--gpus N > 1 outside torchrun: start N replica ranks (one per GPU) with
    torch.distributed.run and return its exit status; a mismatched WORLD_SIZE
    is an error.  Returns None when this process should run the bench itself."""
    ws = os.environ.get("WORLD_SIZE")
    if ws is not None:
        if int(ws) != args.gpus:
            print(json.dumps({"error": f"--gpus {args.gpus} but WORLD_SIZE={ws}"}), flush=True)
            return 2
        return None
    if args.gpus <= 1:
        return None
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
           "--master-port", str(29500 + os.getpid() % 1000), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


# ----------------------------------------------------------------- helpers

_T0 = time.perf_counter()


def progress(what):
    """Elapsed wall time of the bench's phases, on stderr (the JSON line is stdout)."""
    print(f"[bench {time.perf_counter() - _T0:7.1f} s] {what}", file=sys.stderr, flush=True)


def dist_setup(backend=None):
    """Rank, world size; initialises the process group for world size > 1
    (NCCL on GPUs: only the barrier and the max over ranks use it)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return rank, ws


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    """The slowest rank's value (replicas.max_over_ranks over the default group)."""
    if ws == 1:
        return float(x)
    from block_speculative_decoding_ctx_gb300 import replicas
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else None
    return replicas.max_over_ranks(x, dev)


def replica_requests(B, rank, ws):
    """Global request indices [start, stop) of this rank: every rank drafts B
    requests of a job of B * ws (weak scaling), a contiguous slice."""
    from block_speculative_decoding_ctx_gb300 import replicas
    return replicas.partition(B * ws, ws, rank)


def job_value(units_per_rank, ws, ms_max):
    """Whole-job units per second: the units of all ws ranks over the slowest
    rank's time (ms)."""
    from block_speculative_decoding_ctx_gb300 import replicas
    return replicas.job_throughput([units_per_rank] * ws, [ms_max * 1e-3])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during a timed region."""

    def __init__(self):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        dev = os.environ.get("LOCAL_RANK", "0")
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", dev, f"--query-gpu={q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[3:7]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p.get("hbm_gbs", 6800.0), p.get("bf16_tflops", 1900.0), \
            p.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def gpu_weights(dims, seed, dev):
    """Random-init weights of the drafter architecture, N(0, 0.02) bf16, made on the GPU."""
    g = torch.Generator(device=dev).manual_seed(seed)
    d, hd = dims["d"], dims["hd"]

    def mat(r, c):
        return (torch.randn((r, c), generator=g, device=dev) * 0.02).to(torch.bfloat16)

    ones = torch.ones(d, device=dev)
    W = {"embed": mat(dims["vocab"], d), "lm_head": mat(dims["vocab"], d),
         "w_c": mat(d, dims["n_feat"] * dims["feat_dim"]), "g_c": ones, "g_final": ones,
         "layers": []}
    for _ in range(dims["n_layers"]):
        W["layers"].append({"g_attn": ones, "w_qkv": mat((dims["n_q"] + 2 * dims["n_kv"]) * hd, d),
                            "w_o": mat(d, dims["n_q"] * hd), "g_mlp": ones,
                            "w_gate": mat(dims["ffn"], d), "w_up": mat(dims["ffn"], d),
                            "w_down": mat(d, dims["ffn"])})
    return W


def lib_cfg(dims, B, gamma, append_max, topk=4):
    return dict(hidden=dims["d"], n_q_heads=dims["n_q"], n_kv_heads=dims["n_kv"],
                head_dim=dims["hd"], ffn=dims["ffn"], vocab=dims["vocab"],
                n_layers=dims["n_layers"], n_feat=dims["n_feat"], feat_dim=dims["feat_dim"],
                window=dims["window"], gamma_max=max(gamma, 8), topk_max=topk, batch_max=B,
                append_max=append_max, rope_theta=1.0e6, eps=1.0e-6, mask_id=-1)


def time_graph(g, steps, stream):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / steps


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    # work queued on other streams (workspace fills, a prefill) must land first
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        fn()                    # eager warm-up outside the capture
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


# ------------------------------------------------------------- GPU cycle

SAMPLING_T, SAMPLING_TOP_P = 0.7, 0.99     # model card, section "Acceptance length"


class Cycle:
    """State and launch sequence of one speculative cycle for B requests.

    lens: context length of each request; the last min(L, W) positions are
    appended before timing (the ring wraps for L > W).  A step is
      ctx_append   features of the positions the last verification committed
      draft_block  greedy (top-1 drafts) or sampled (q, y ~ q at T, top-p)
      stand-in     target logits = draft logits + N(0, sigma), the last row
                   repeated for the bonus position (excluded from the timing)
      probs        p = top_p(softmax(target / T))              (sampled only)
      verify       greedy or sampled; writes the next anchor and append count
    """

    def __init__(self, dfl, h, dims, B, gamma, lens, sigma, dev, seed, sampled=False, topk=4,
                 req0=0):
        self.dfl, self.h, self.dims, self.B, self.gamma = dfl, h, dims, B, gamma
        self.sampled, self.topk = sampled, topk
        V, Wn = dims["vocab"], dims["window"]
        G = gamma - 1
        gen = torch.Generator(device=dev).manual_seed(seed)
        shape = (dims["n_layers"], B, dims["n_kv"], Wn, dims["hd"])
        self.rk = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        self.rv = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        self.ws_a = dfl.workspace(dfl.dflash_append_workspace_bytes(h), dev)
        self.ws_d = dfl.workspace(dfl.dflash_draft_workspace_bytes(h), dev)
        self.ws_v = dfl.workspace(dfl.dflash_verify_workspace_bytes(B, gamma, V), dev)
        lens = torch.as_tensor(lens, dtype=torch.int64)
        n0 = torch.clamp(lens, max=Wn)
        self.ctx = (lens - n0).to(dev)
        if int(n0.max()) > 0:
            feats0 = torch.randn((B, int(n0.max()), dims["n_feat"], dims["feat_dim"]), generator=gen,
                                 device=dev).to(torch.bfloat16)
            dfl.dflash_ctx_append(h, feats0, n0.to(torch.int32).to(dev), self.ctx, self.rk, self.rv,
                                  self.ws_a)
            del feats0
        self.feats = torch.randn((B, gamma, dims["n_feat"], dims["feat_dim"]), generator=gen,
                                 device=dev).to(torch.bfloat16)
        self.anchor = torch.randint(0, V - 1, (B,), generator=gen, device=dev, dtype=torch.int32)
        self.n_app = torch.ones(B, dtype=torch.int32, device=dev)
        self.noise = torch.randn((B, gamma, V), generator=gen, device=dev) * sigma
        self.logits = torch.empty((B, G, V), device=dev)
        self.ids = torch.empty((B, G, topk), dtype=torch.int32, device=dev)
        self.vals = torch.empty((B, G, topk), device=dev)
        self.lse = torch.empty((B, G), device=dev)
        self.draft = torch.empty((B, G), dtype=torch.int32, device=dev)
        self.target = torch.empty((B, gamma, V), device=dev)
        self.acc = torch.empty(B, dtype=torch.int32, device=dev)
        self.tok = torch.empty((B, gamma), dtype=torch.int32, device=dev)
        self.tau_sum = torch.zeros(B, dtype=torch.int64, device=dev)
        self.out = dict(topk_ids=self.ids, topk_vals=self.vals, lse=self.lse, logits=self.logits,
                        draft=self.draft)
        self.sampling = None
        torch.cuda.synchronize()   # the prefill and workspace fills ran on the current stream
        if sampled:
            from block_speculative_decoding_ctx_gb300 import synth
            self.seeds = synth.seeds(B + req0, seed)[req0:].to(dev)   # Philox key per request
            self.q = torch.empty((B, G, V), device=dev)
            self.p = torch.empty((B, gamma, V), device=dev)
            self.ws_p = dfl.workspace(dfl.dflash_probs_workspace_bytes(B * gamma, V), dev)
            self.out["q"] = self.q
            self.sampling = dict(temperature=SAMPLING_T, top_p=SAMPLING_TOP_P, seeds=self.seeds, step=1)
            torch.cuda.synchronize()

    def append(self):
        self.dfl.dflash_ctx_append(self.h, self.feats, self.n_app, self.ctx, self.rk, self.rv, self.ws_a)

    def draft_pass(self):
        self.dfl.dflash_draft_block(self.h, self.anchor, self.ctx, self.rk, self.rv, self.gamma,
                                    self.ws_d, topk=self.topk, out=self.out, sampling=self.sampling)

    def stand_in(self):
        G = self.gamma - 1
        torch.add(self.logits, self.noise[:, :G], out=self.target[:, :G])
        torch.add(self.logits[:, G - 1], self.noise[:, G], out=self.target[:, G])
        if self.sampled:
            self.seeds.add_(1)          # fresh Philox streams every cycle of a replayed graph

    def prep(self):
        if self.sampled:
            self.dfl.dflash_probs(self.target, SAMPLING_T, SAMPLING_TOP_P, self.p, self.ws_p)

    def verify(self):
        if self.sampled:
            self.dfl.dflash_verify(self.dfl.DFLASH_VERIFY_SAMPLED, self.p, self.draft, self.acc, self.tok,
                                   self.ws_v, q=self.q, seeds=self.seeds, step=1,
                                   next_anchor=self.anchor, n_append=self.n_app)
        else:
            self.dfl.dflash_verify(self.dfl.DFLASH_VERIFY_GREEDY, self.target, self.draft, self.acc,
                                   self.tok, self.ws_v, next_anchor=self.anchor, n_append=self.n_app)
        self.tau_sum.add_(self.n_app)

    def step(self):
        self.append()
        self.draft_pass()
        self.stand_in()
        self.prep()
        self.verify()


# DRAM bytes (read + written) of the draft pass's GEMM launches at batch 1,
# gamma 8, five layers, from ncu's dram__bytes_read.sum + dram__bytes_write.sum
# of a one-layer pass (the layer's four launches scaled to five layers, plus
# the LM head), or None when the GEMM kernels have changed since the counters
# were taken.  The last capture (4,882.1 MB against 4,871,884,288 algorithmic
# bytes) predates the split-K reduction's asynchronous-copy landing.
GEMM_TRAFFIC_PER_PASS = None


def gpu_launches_per_step(dims, tokens, with_append=True, sampled=False):
    # QKV, attention, O, RMSNorm, gate|up, down, RMSNorm; up to 32 tokens the
    # RMSNorms run inside the GEMMs that consume them
    per_layer = 5 if tokens <= 32 else 7
    n = 1 + per_layer * dims["n_layers"] + 2          # embed+norm, layers, LM head, top-k
    n += 1                                            # verify
    if sampled:
        n += 3                                        # q, y ~ q, p of the target
    if with_append:
        n += 4                                        # W_c GEMM, RMSNorm, K/V GEMM, lengths
    return n


def acceptance_stats(cyc, g_step, stream, B, G, steps, sigma):
    """Accepted lengths over untimed replays of the cycle: the distribution of
    tau (accepted drafts + 1), the rate at which draft position i is accepted
    (tau >= i + 1), and that rate given position i - 1 was accepted (the decay
    along the block)."""
    dev = cyc.n_app.device
    hist = torch.zeros(G + 1, dtype=torch.int64, device=dev)
    ones = torch.ones(B, dtype=torch.int64, device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(steps):
            g_step.replay()
            hist.scatter_add_(0, cyc.n_app.long(), ones)
    stream.synchronize()
    out = {"cycles": steps, "requests_per_cycle": B, "sigma": sigma}
    out.update(acceptance_rates(hist.cpu().tolist(), G))
    return out


def acceptance_rates(h, G):
    """From a histogram h[tau] (tau = 1..G): the mean, the rate at which draft
    position i = 1..G-1 is accepted (tau >= i + 1) and that rate given that
    position i - 1 was accepted."""
    n = max(sum(h), 1)
    at_least = [sum(h[t] for t in range(i + 1, G + 1)) / n for i in range(1, G)]
    given = [at_least[0]] + [at_least[i] / at_least[i - 1] if at_least[i - 1] > 0 else None
                             for i in range(1, G - 1)]
    return {"tau_hist": list(h), "tau_mean": round(sum(t * c for t, c in enumerate(h)) / n, 3),
            "accept_rate_by_position": [round(a, 4) for a in at_least],
            "accept_rate_given_previous": [None if g is None else round(g, 4) for g in given]}


def pass_profile(dfl, h, fn, stream, passes, run=3):
    """Per-launch device times of the draft pass inside a replayed graph: the
    library's completion marks charge every launch the time from the previous
    launch's completion to its own, so the launches add up to the pass.  The
    graph is replayed `run` times back to back and the last replay's marks are
    read, as the timed loops replay it (the first launch is then charged from
    the previous replay's end, not from a graph launch)."""
    dfl.dflash_profile_enable(h, 128)
    g = capture(fn, stream)
    rows = []
    with torch.cuda.stream(stream):
        for _ in range(passes):
            for _ in range(run):
                g.replay()
            stream.synchronize()
            rows.append(dfl.dflash_profile_read(h))
    dfl.dflash_profile_enable(h, 0)
    del g
    n = len(rows)
    kinds = {}
    for rr in rows:
        for r in rr:
            kinds[r[2]] = kinds.get(r[2], 0.0) + r[0] / n
    return rows, kinds


def draft_flops(dims, B, G):
    """Algorithmic FLOPs of the draft pass's GEMMs (2 per multiply-add)."""
    M = B * G
    d, F, V = dims["d"], dims["ffn"], dims["vocab"]
    qkv = (dims["n_q"] + 2 * dims["n_kv"]) * dims["hd"]
    f = dims["n_layers"] * 2.0 * M * d * (qkv + dims["n_q"] * dims["hd"] + 3 * F)
    return f + 2.0 * B * (G - 1) * d * V


def run_ours(args, rank, ws):
    import block_speculative_decoding_ctx_gb300 as dfl
    dfl.lib()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    dims = dict(DIMS_FULL, n_layers=args.layers)
    B, G = args.batch, args.gamma
    W = gpu_weights(dims, 1234, dev)
    cfg = lib_cfg(dims, max(B, 1), G, max(min(args.context, dims["window"]), G))
    if args.profile_cycles and args.weights == "e4m3":
        h = dfl.dflash_create(dict(cfg, weight_format=dfl.DFLASH_WEIGHTS_E4M3), dfl.quantize_weights_e4m3(W))
    else:
        h = dfl.dflash_create(cfg, W)
    r0, _ = replica_requests(B, rank, ws)
    cyc = Cycle(dfl, h, dims, B, G, [args.context] * B, args.sigma, dev, 99 + r0,
                sampled=bool(args.profile_cycles and args.sampled))
    stream = torch.cuda.Stream(device=dev)
    if args.profile_cycles:
        with torch.cuda.stream(stream):
            for _ in range(args.profile_cycles):
                cyc.step()
        torch.cuda.synchronize()
        return {"profile_cycles": args.profile_cycles, "layers": args.layers,
                "tau_sum": int(cyc.tau_sum.sum().item())}

    g_step = capture(cyc.step, stream)
    g_stand = capture(cyc.stand_in, stream)
    g_draft = capture(cyc.draft_pass, stream)
    g_app = capture(cyc.append, stream)
    g_ver = capture(cyc.verify, stream)
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            g_step.replay()
    torch.cuda.synchronize()
    cyc.tau_sum.zero_()

    # ------------------------------------------------------ timed region
    barrier(ws)
    torch.cuda.synchronize()
    clocks = ClockSampler()
    t_step = time_graph(g_step, args.steps, stream)
    tau_mean = cyc.tau_sum.sum().item() / (args.steps * B)
    clk = clocks.stop()
    barrier(ws)
    t_stand = time_graph(g_stand, args.steps, stream)
    t_draft = time_graph(g_draft, args.steps, stream)
    t_app = time_graph(g_app, args.steps, stream)
    t_ver = time_graph(g_ver, args.steps, stream)
    t_path = max(t_step - t_stand, 1e-6)
    t_path_max = max_over_ranks(t_path, ws)

    # -------------------------- acceptance along the block (untimed replays)
    progress("headline timed")
    acceptance = acceptance_stats(cyc, g_step, stream, B, G, max(64, 256 // B), args.sigma)

    # ------------------------------------ dominant kernel (GEMMs of the pass)
    rows, kinds = pass_profile(dfl, h, cyc.draft_pass, stream, args.steps)
    n_pass = len(rows)
    gemm = [r for r in rows[0] if r[2] == "gemm"]
    ms = sum(r[0] for rr in rows for r in rr if r[2] == "gemm") / n_pass
    by = sum(r[1] for r in gemm)
    lm = [[r for r in rr if r[2] == "gemm"][-1] for rr in rows]
    hbm, tf, tf_sus, src = measured_peaks()
    achieved = by / (ms * 1e-3) / 1e9
    roof = {"kernel": f"gemm_tc_kernel (all {len(gemm)} GEMM launches of the draft pass)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "peak_source": src,
            "traffic": (GEMM_TRAFFIC_PER_PASS if (B, G, args.layers) == (1, 8, 5) else None),
            "traffic_note": "null: the GEMM kernel changed after the last DRAM counters "
                            "(4,882.1 MB per pass, 1.002x of algorithmic)" if GEMM_TRAFFIC_PER_PASS is None
                            else "one-layer ncu capture scaled to five layers",
            "traffic_unit": "DRAM bytes read + written per pass (all GEMM launches)",
            "gemm_ms_per_pass": round(ms, 4), "gemm_bytes_per_pass": by,
            "timing": "completion-to-completion intervals of each launch inside a replayed graph "
                      "of the draft pass (library completion marks); the launches of a pass add "
                      "up to profiled_pass_ms",
            "profiled_pass_ms": round(sum(kinds.values()), 4),
            "lm_head_GBps": round(lm[0][1] / (statistics.median(r[0] for r in lm) * 1e-3) / 1e9, 1),
            "kernel_ms_per_pass_by_kind": {k: round(v, 4) for k, v in kinds.items()},
            "first_layer_launches": [[r[2], round(r[0] * 1e3, 1), round(r[1] / (r[0] * 1e-3) / 1e9, 1)]
                                     for r in rows[-1][:9]]}

    # ------------------------------------------------- end to end (host buffers)
    progress("acceptance and launch profile")
    e2e = run_e2e(args, dfl, cyc, stream, g_step)
    progress("end to end")

    extras, sweep, fp8 = {}, None, None
    if not args.no_extras and ws == 1:
        del cyc, g_step, g_stand, g_draft, g_app, g_ver, h
        torch.cuda.empty_cache()
        fp8 = run_fp8_line(args, dfl, dims, W, dev, stream)
        progress("E4M3 line")
        torch.cuda.empty_cache()
        extras = run_batch_lines(args, dfl, dims, W, dev, stream)
        progress("batch lines")
        del W
        torch.cuda.empty_cache()
        sweep = verify_sweep(args, dfl, dev, stream)
        progress("verify sweep")

    value = job_value(B, ws, t_path_max)
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "draft blocks/s",
        "n_gpus": ws, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(t_path_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic (random-init weights N(0,0.02), "
        "features N(0,1), target logits = draft logits + N(0,sigma))",
        "config": {"workload": WORKLOAD.format(B=B, G=G, L=args.context), "batch": B, "gamma": G,
                   "context": args.context, "sigma": args.sigma,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": "inputs larger than L2: 4.9 GB of weights streamed per step"},
        "verified_tokens_per_s": round(job_value(tau_mean * B, ws, t_path_max), 2),
        "tau_mean": round(tau_mean, 3),
        "stage_ms": {"ctx_append": round(t_app, 4), "draft_block": round(t_draft, 4),
                     "verify": round(t_ver, 4), "target_stand_in_excluded": round(t_stand, 4)},
        "clocks": clk, "e2e": e2e,
        "gpu_launches": gpu_launches_per_step(dims, B * G) * args.steps,
        "roofline": roof,
        "acceptance": acceptance,
    }
    if extras:
        res["batches"] = extras
    if sweep:
        res["verify_sweep"] = sweep
    if fp8:
        res["e4m3_weights"] = fp8
    return res


def run_fp8_line(args, dfl, dims, W, dev, stream):
    """The headline cycle (batch 1, gamma 8, context 4,096, greedy) on E4M3
    weights made on the device from the same bf16 weights
    (dflash_quantize_e4m3): half the weight bytes per draft pass."""
    try:
        Wq = dfl.quantize_weights_e4m3(W)
        cfg = dict(lib_cfg(dims, 1, 8, dims["window"]), weight_format=dfl.DFLASH_WEIGHTS_E4M3)
        h = dfl.dflash_create(cfg, Wq)
        cyc = Cycle(dfl, h, dims, 1, 8, [4096], args.sigma, dev, 99)
        g_step = capture(cyc.step, stream)
        g_stand = capture(cyc.stand_in, stream)
        g_draft = capture(cyc.draft_pass, stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g_step.replay()
        torch.cuda.synchronize()
        cyc.tau_sum.zero_()
        steps = max(5, args.steps)
        t_step = time_graph(g_step, steps, stream)
        tau = cyc.tau_sum.sum().item() / steps
        t_path = max(t_step - time_graph(g_stand, steps, stream), 1e-6)
        t_draft = time_graph(g_draft, steps, stream)
        rows, kinds = pass_profile(dfl, h, cyc.draft_pass, stream, 5)
        gemm = [r for r in rows[-1] if r[2] == "gemm"]
        by = sum(r[1] for r in gemm)
        gemm_ms = kinds.get("gemm", 0.0)
        hbm = measured_peaks()[0]
        res = {"workload": "full dims, batch 1, gamma 8, context 4096, top-4, greedy verify; drafter "
                           "matrices and LM head E4M3 with float32 row scales (quantized on the device)",
               "draft_blocks_per_s": round(1000.0 / t_path, 2), "ms_per_step": round(t_path, 4),
               "verified_tokens_per_s": round(tau * 1000.0 / t_path, 2), "tau_mean": round(tau, 3),
               "draft_block_ms": round(t_draft, 4),
               "gemm_bytes_per_pass": by, "gemm_ms_per_pass": round(gemm_ms, 4),
               "gemm_GBps": round(by / (gemm_ms * 1e-3) / 1e9, 1),
               "gemm_frac_of_hbm": round(by / (gemm_ms * 1e-3) / 1e9 / hbm, 4),
               "kernel_ms_per_pass_by_kind": {k: round(v, 4) for k, v in kinds.items()},
               "first_layer_launches_us_GBps": [[r[2], round(r[0] * 1e3, 1), round(r[1] / (r[0] * 1e-3) / 1e9, 1)]
                                                for r in rows[-1][:9]] +
                                               [["lm_head", round(gemm[-1][0] * 1e3, 1),
                                                 round(gemm[-1][1] / (gemm[-1][0] * 1e-3) / 1e9, 1)]],
               "status": dfl.dflash_read_status(cyc.ws_d)}
        del h, cyc, g_step, g_stand, g_draft, Wq
        return res
    except Exception as e:  # keep the headline line; report the failure in place
        return {"error": f"{type(e).__name__}: {e}"}


def run_e2e(args, dfl, cyc, stream, g_step):
    """The same cycle through the public API with pinned host inputs and
    outputs: features and stand-in target noise copied in, accept length and
    tokens copied out, every step, host timer around the whole loop.  The
    cycle's calls are captured once in a CUDA graph (the API supports capture,
    as a serving loop would use it) and replayed; the eager variant (every
    call made each step) is reported beside it."""
    B, G, V = cyc.B, cyc.gamma, cyc.dims["vocab"]
    feats_h = cyc.feats.cpu().pin_memory()
    noise_h = cyc.noise.cpu().pin_memory()
    acc_h = torch.empty(B, dtype=torch.int32).pin_memory()
    tok_h = torch.empty((B, G), dtype=torch.int32).pin_memory()
    steps = max(5, args.steps // 2)

    def one(graph):
        cyc.feats.copy_(feats_h, non_blocking=True)
        cyc.noise.copy_(noise_h, non_blocking=True)
        if graph:
            g_step.replay()
        else:
            cyc.step()
        acc_h.copy_(cyc.acc, non_blocking=True)
        tok_h.copy_(cyc.tok, non_blocking=True)

    def timed(graph):
        with torch.cuda.stream(stream):
            for _ in range(3):
                one(graph)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(steps):
                one(graph)
                stream.synchronize()          # the caller reads the result every step
            return (time.perf_counter() - t0) / steps

    t_graph, t_eager = timed(True), timed(False)
    h2d = feats_h.numel() * feats_h.element_size() + noise_h.numel() * noise_h.element_size()
    d2h = acc_h.numel() * 4 + tok_h.numel() * 4
    return {"value": round(B / t_graph, 2), "unit": "draft blocks/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(t_graph * 1e3, 4),
            "eager": {"value": round(B / t_eager, 2), "ms_per_step": round(t_eager * 1e3, 4)},
            "note": "host copies in and out every step around a replay of the captured cycle "
                    "(ctx_append, draft_block, stand-in target, verify); 'eager' makes every "
                    "API call each step instead"}


def attention_ring_bytes(dims, B, context):
    """Ring K/V bytes the draft pass's attention reads: every layer, request and
    KV head streams its visible window (min(context, W) keys) of bf16 K and V."""
    keys = min(context, dims["window"])
    return dims["n_layers"] * B * dims["n_kv"] * keys * dims["hd"] * 2 * 2


# Batch workloads of the metric besides the headline (name, B, gamma, contexts,
# sampled verification, stand-in noise sigma; None = the --sigma of greedy lines).
BATCH_LINES = (
    ("batch16_gamma8_sampled", 16, 8, "loguniform", True, 1.0),
    ("batch32_gamma8_greedy", 32, 8, 8192, False, None),
    ("batch32_gamma8_sampled", 32, 8, 8192, True, 1.0),
    ("batch32_gamma16_greedy", 32, 16, 8192, False, None),
)


def batch_contexts(spec, B):
    """Context lengths of a batch line: a fixed length, or log-uniform in
    512 .. 131,072 (the model card's long-context range; the ring keeps the
    last 4,096 positions)."""
    if spec == "loguniform":
        from block_speculative_decoding_ctx_gb300 import synth
        return synth.log_uniform_lengths(B, 512, 131072, 80)
    return torch.full((B,), int(spec), dtype=torch.int64)


def run_batch_lines(args, dfl, dims, W, dev, stream):
    out = {}
    hbm, tf, tf_sus, src = measured_peaks()
    for name, B, G, ctx_spec, sampled, sigma in BATCH_LINES:
        try:
            out[name] = run_batch_line(args, dfl, dims, W, dev, stream, B, G, ctx_spec, sampled,
                                       args.sigma if sigma is None else sigma, hbm, tf_sus, src)
        except Exception as e:  # keep the headline line; report the failure in place
            out[name] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
    return out


def run_batch_line(args, dfl, dims, W, dev, stream, B, G, ctx_spec, sampled, sigma, hbm, tf_sus, src):
    """One batch workload as a whole cycle (see Cycle): draft blocks/s and
    verified tokens/s of the step, the time of each stage, and the draft
    pass's GEMM and attention rates from its launch profile."""
    lens = batch_contexts(ctx_spec, B)
    h = dfl.dflash_create(lib_cfg(dims, B, G, dims["window"]), W)
    cyc = Cycle(dfl, h, dims, B, G, lens, sigma, dev, 7 + B + G, sampled=sampled)
    g_step = capture(cyc.step, stream)
    g_stand = capture(cyc.stand_in, stream)
    g_draft = capture(cyc.draft_pass, stream)
    g_app = capture(cyc.append, stream)
    g_prep = capture(cyc.prep, stream) if sampled else None
    g_ver = capture(cyc.verify, stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g_step.replay()
    torch.cuda.synchronize()
    cyc.tau_sum.zero_()
    steps = max(5, args.steps // 2)
    t_step = time_graph(g_step, steps, stream)
    tau = cyc.tau_sum.sum().item() / (steps * B)
    t_stand = time_graph(g_stand, steps, stream)
    stage = {"ctx_append": time_graph(g_app, steps, stream),
             "draft_block": time_graph(g_draft, steps, stream)}
    if sampled:
        stage["probs_target"] = time_graph(g_prep, steps, stream)
    stage["verify"] = time_graph(g_ver, steps, stream)
    stage = {k: round(v, 4) for k, v in stage.items()}
    stage["target_stand_in_excluded"] = round(t_stand, 4)
    t_path = max(t_step - t_stand, 1e-6)
    status = {"ctx_append": dfl.dflash_read_status(cyc.ws_a), "draft_block": dfl.dflash_read_status(cyc.ws_d),
              "verify": dfl.dflash_read_status(cyc.ws_v)}
    rows, kinds = pass_profile(dfl, h, cyc.draft_pass, stream, 3)
    prof = rows[-1]
    gemm_ms = kinds.get("gemm", 0.0)
    attn_ms = kinds.get("attention", 0.0)
    gemm_tflops = draft_flops(dims, B, G) / (gemm_ms * 1e-3) / 1e12
    M = B * G
    d, F, V = dims["d"], dims["ffn"], dims["vocab"]
    qkv = (dims["n_q"] + 2 * dims["n_kv"]) * dims["hd"]
    qd = dims["n_q"] * dims["hd"]
    fl = [2.0 * M * d * qkv, 2.0 * M * d * qd, 2.0 * M * d * 2 * F, 2.0 * M * F * d]
    gl = [p for p in prof if p[2] == "gemm"]
    layer0 = [[n, round(p[0] * 1e3, 1), round(f / (p[0] * 1e-3) / 1e12, 1)]
              for n, p, f in zip(("qkv", "o", "gate_up", "down"), gl[:4], fl)]
    layer0.append(["lm_head", round(gl[-1][0] * 1e3, 1),
                   round(2.0 * B * (G - 1) * d * V / (gl[-1][0] * 1e-3) / 1e12, 1)])
    ring = sum(attention_ring_bytes(dims, 1, int(L)) for L in lens)
    attn_gbps = ring / (attn_ms * 1e-3) / 1e9
    res = {"batch": B, "gamma": G,
           "contexts": ("log-uniform 512..131072 (seed 80), ring holds the last 4096"
                        if ctx_spec == "loguniform" else f"{ctx_spec} (window 4096)"),
           "verification": (f"sampled, T={SAMPLING_T}, top-p {SAMPLING_TOP_P}" if sampled else "greedy"),
           "sigma": sigma,
           "draft_blocks_per_s": round(B * 1000.0 / t_path, 2),
           "verified_tokens_per_s": round(tau * B * 1000.0 / t_path, 2),
           "tau_mean": round(tau, 3), "ms_per_step": round(t_path, 4), "stage_ms": stage,
           "gemm_ms": round(gemm_ms, 4), "attention_ms": round(attn_ms, 4),
           "kernel_ms_per_pass_by_kind": {k: round(v, 4) for k, v in kinds.items()},
           "attention_ring_GBps": round(attn_gbps, 1),
           "attention_frac_of_hbm": round(attn_gbps / hbm, 4),
           "gemm_tflops": round(gemm_tflops, 1),
           "gemm_frac_of_tensor_peak": round(gemm_tflops / tf_sus, 4),
           "first_layer_gemms_us_tflops": layer0,
           "peak_tflops_sustained": tf_sus, "peak_source": src,
           "peak_note": "fp16 operands; the measured bf16 peak stands for fp16 "
                        "(nominal dense rates equal)",
           "status": status}
    del h, cyc, g_step, g_stand, g_draft, g_app, g_prep, g_ver
    return res


# Verify-only sweep: batch x gamma x noise of the target around the draft.
SWEEP_B = (1, 16, 64, 256)
SWEEP_GAMMA = (8, 16)
SWEEP_SIGMA = (0.25, 1.0, 4.0)


def sampled_verify_bytes(n, G, V):
    """Algorithmic bytes of one sampled verification: the accept tests read
    p_i(y_i) and q_i(y_i) of the n accepted drafts and of the rejected one;
    a rejection at position n < G reads the rows p_n and q_n for the residual,
    an all-accepted block reads the bonus row p_G; outputs are the accept
    length and gamma tokens."""
    n = [int(x) for x in n]
    tests = sum(8 * (k + (1 if k < G else 0)) for k in n)
    rows = sum(8 * V if k < G else 4 * V for k in n)
    return tests + rows + len(n) * 4 * (G + 2)


def verify_sweep(args, dfl, dev, stream):
    """dflash_verify alone over fp32 p and q of the full vocabulary: draft
    logits N(0, 3), target logits = draft + N(0, sigma), p and q their softmax,
    y ~ q drawn by dflash_sample_draft.  Each call is timed with CUDA events
    after an L2 flush (a 256 MiB write), so small batches read from HBM too.
    GB/s = algorithmic bytes (sampled_verify_bytes; greedy: gamma target rows
    per request) / time."""
    hbm = measured_peaks()[0]
    V = DIMS_FULL["vocab"]
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)
    reps = 5
    rows = []

    def time_calls(fn):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        torch.cuda.synchronize()        # inputs were made on the current stream
        with torch.cuda.stream(stream):
            fn()
            for e0, e1 in ev:
                flush.zero_()
                e0.record(stream)
                fn()
                e1.record(stream)
        stream.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)

    for B in SWEEP_B:
        for gamma in SWEEP_GAMMA:
            G = gamma - 1
            gen = torch.Generator(device=dev).manual_seed(1000 + B + gamma)
            d = torch.randn((B, gamma, V), generator=gen, device=dev) * 3.0
            q = torch.softmax(d[:, :G], dim=-1)
            seeds = torch.randint(0, 2 ** 62, (B,), generator=gen, device=dev, dtype=torch.int64)
            y = torch.empty((B, G), dtype=torch.int32, device=dev)
            ws_s = dfl.workspace(dfl.dflash_sample_workspace_bytes(B * G, V), dev)
            ws_v = dfl.workspace(dfl.dflash_verify_workspace_bytes(B, gamma, V), dev)
            n = torch.empty(B, dtype=torch.int32, device=dev)
            tok = torch.empty((B, gamma), dtype=torch.int32, device=dev)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                dfl.dflash_sample_draft(q, seeds, 3, y, ws_s)
            torch.cuda.synchronize()
            for sigma in SWEEP_SIGMA:
                t = d + torch.randn((B, gamma, V), generator=gen, device=dev) * sigma
                p = torch.softmax(t, dim=-1)
                del t
                ms = time_calls(lambda: dfl.dflash_verify(dfl.DFLASH_VERIFY_SAMPLED, p, y, n, tok, ws_v,
                                                          q=q, seeds=seeds, step=3))
                acc = n.cpu()
                by = sampled_verify_bytes(acc.tolist(), G, V)
                rows.append({"mode": "sampled", "batch": B, "gamma": gamma, "sigma": sigma,
                             "us": round(ms * 1e3, 2), "GBps": round(by / (ms * 1e-3) / 1e9, 1),
                             "frac_of_hbm": round(by / (ms * 1e-3) / 1e9 / hbm, 4),
                             "tau_mean": round(float(acc.float().mean()) + 1.0, 3)})
                del p
            ms = time_calls(lambda: dfl.dflash_verify(dfl.DFLASH_VERIFY_GREEDY, d, y, n, tok, ws_v))
            by = 4.0 * B * gamma * V
            rows.append({"mode": "greedy", "batch": B, "gamma": gamma, "us": round(ms * 1e3, 2),
                         "GBps": round(by / (ms * 1e-3) / 1e9, 1),
                         "frac_of_hbm": round(by / (ms * 1e-3) / 1e9 / hbm, 4)})
            del d, q, y, ws_s, ws_v
            torch.cuda.empty_cache()
    return {"vocab": V, "recipe": "draft logits N(0,3); target = draft + N(0,sigma); p, q = softmax; "
                                  "y ~ q; one call per timing after a 256 MiB L2 flush, median of "
                                  f"{reps}", "peak_GBps": hbm, "points": rows}


# --------------------------------------------------------------- CPU oracle

class OracleCycle:
    """One speculative cycle of one request, computed by the float64 CPU
    oracle: ctx_append of the positions the last cycle committed (W_c fusion
    and the K/V of every layer), the block draft over a full window with the
    full LM head and top-4, and greedy verification.  At the full dimensions
    the five layers share one random weight set (the work is the same as five
    distinct ones; generating 1.65 B random parameters on the host would take
    longer than the cycles themselves)."""

    def __init__(self, dims, gamma=8, seed=5):
        import numpy as np

        from block_speculative_decoding_ctx_gb300 import synth
        from oracle import model as om
        self.np, self.om, self.gamma = np, om, gamma
        d = dims["d"]
        g = synth.gen(seed)

        def mat(r, c):
            return (torch.randn((r, c), generator=g) * 0.02).to(torch.bfloat16)

        head = mat(dims["vocab"], d)
        layer = {"g_attn": torch.ones(d), "w_qkv": mat((dims["n_q"] + 2 * dims["n_kv"]) * dims["hd"], d),
                 "w_o": mat(d, dims["n_q"] * dims["hd"]), "g_mlp": torch.ones(d),
                 "w_gate": mat(dims["ffn"], d), "w_up": mat(dims["ffn"], d),
                 "w_down": mat(d, dims["ffn"])}
        self.W = {"embed": head, "lm_head": head, "g_final": torch.ones(d), "g_c": torch.ones(d),
                  "w_c": mat(d, dims["n_feat"] * dims["feat_dim"]), "layers": [layer] * dims["n_layers"]}
        self.cfg = om.Config(**dims)
        shape = (dims["n_layers"], 1, dims["n_kv"], dims["window"], dims["hd"])
        self.rk = torch.randn(shape, generator=g).to(torch.bfloat16).double().numpy()
        self.rv = torch.randn(shape, generator=g).to(torch.bfloat16).double().numpy()
        self.n_app = max(1, gamma - 3)
        self.feats = torch.randn((self.n_app, dims["n_feat"], dims["feat_dim"]),
                                 generator=g).to(torch.bfloat16)
        self.L = 2 * dims["window"]
        self.noise = np.random.default_rng(seed).normal(0, 0.05, (1, gamma, dims["vocab"])).astype(np.float32)

    def run(self):
        from oracle import verify as over
        np, om = self.np, self.om
        t0 = time.perf_counter()
        om.ctx_append(self.cfg, self.W, self.rk, self.rv, 0, self.feats, self.L)
        self.L += self.n_app
        out = om.draft_pass(self.cfg, self.W, self.rk, self.rv, np.array([self.L]), np.array([3]),
                            self.gamma)
        logits = out["logits"]
        om.topk(logits[0], 4)
        om.logsumexp(logits)
        tgt = np.concatenate([logits, logits[:, -1:]], axis=1).astype(np.float32) + self.noise
        over.greedy(tgt, logits.argmax(-1))
        return time.perf_counter() - t0


SAMPLE = ("whole speculative cycles of one request at the full dimensions (ctx_append of 5 "
          "positions, 5-layer block draft over a 4,096 window with the full LM head and top-4, "
          "greedy verify), float64 numpy oracle")
DIMS_TINY = dict(d=256, n_q=4, n_kv=2, hd=64, ffn=512, vocab=1024, n_layers=1, n_feat=5,
                 feat_dim=256, window=64)


def oracle_rate(oc, target_s):
    """Cycles per second of an OracleCycle over about target_s seconds."""
    oc.run()                                  # warm-up (page-in, BLAS threads)
    times = []
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < target_s or len(times) < 2:
        times.append(oc.run())
    return 1.0 / statistics.mean(times), len(times), sum(times)


def oracle_verify_rate(B, target_s=1.0, gamma=8, sigma=1.0):
    """Requests per second of the oracle's sampled verification over the full
    vocabulary (the verify-sweep recipe: draft logits N(0, 3), target = draft
    + N(0, sigma), p and q their softmax, y ~ q)."""
    import numpy as np

    from oracle import verify as over
    V = DIMS_FULL["vocab"]
    g = torch.Generator().manual_seed(500 + B)
    d = torch.randn((B, gamma, V), generator=g) * 3.0
    p = torch.softmax(d + torch.randn((B, gamma, V), generator=g) * sigma, dim=-1).numpy()
    q = torch.softmax(d[:, :gamma - 1], dim=-1).numpy()
    seeds = np.arange(B, dtype=np.uint64) + np.uint64(77)
    y = torch.multinomial(torch.from_numpy(q).reshape(-1, V), 1, generator=g).reshape(B, gamma - 1).numpy()
    times = []
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < target_s or not times:
        t0 = time.perf_counter()
        over.sampled(p, q, y, seeds, 3)
        times.append(time.perf_counter() - t0)
    return B / statistics.mean(times)


def cpu_probe(kind):
    """One oracle timing, for a child process whose BLAS runs on one thread."""
    if kind == "tiny":
        r, n, _ = oracle_rate(OracleCycle(dict(DIMS_TINY), gamma=4), 2.0)
        return {"tiny_cycles_per_s": round(r, 2), "cycles": n}
    return {"verify16_requests_per_s": round(oracle_verify_rate(16), 2)}


def one_core(kind):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    env.pop("WORLD_SIZE", None)
    try:
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-probe", kind],
                             env=env, capture_output=True, text=True, timeout=120)
        return json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as e:  # report in place; the GPU line stands
        return {"error": f"{type(e).__name__}: {e}"}


def cpu_baseline(target_s=12.0):
    value, n, total = oracle_rate(OracleCycle(dict(DIMS_FULL)), target_s)
    tiny, n_tiny, _ = oracle_rate(OracleCycle(dict(DIMS_TINY), gamma=4), 2.0)
    verify = {f"batch{B}": round(oracle_verify_rate(B), 2) for B in (1, 16, 256)}
    return {"value": round(value, 5), "unit": "draft blocks/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{n} {SAMPLE}; {total:.1f} s of CPU work",
            "tiny_config": {"draft_blocks_per_s": round(tiny, 2), "cores": os.cpu_count(),
                            "sample": f"{n_tiny} tiny-config cycles (1 layer, hidden 256, gamma 4, "
                                      "window 64, vocabulary 1,024; append 1 position, draft, "
                                      "greedy verify)",
                            "one_core": one_core("tiny")},
            "verify_sweep": {"unit": "requests/s (sampled verification, gamma 8, sigma 1, "
                                     "vocabulary 151,936)", "cores": os.cpu_count(), **verify,
                             "one_core": one_core("verify16")}}


def run_reference(args, rank, ws):
    if rank != 0:
        return None
    oc = OracleCycle(dict(DIMS_FULL))
    warm = max(args.warmup, 3)
    for _ in range(warm):
        oc.run()
    times = [oc.run() for _ in range(args.steps)]
    t = statistics.mean(times)
    value = 1.0 / t
    return {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "draft blocks/s",
            "n_gpus": ws, "steps": args.steps, "warmup": warm, "ms_per_step": round(t * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD.format(B=1, G=8, L=4096) +
                                            " (float64 CPU oracle)", "batch": 1, "gamma": 8},
            "cpu_baseline": {"value": round(value, 5), "unit": "draft blocks/s",
                             "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{args.steps} timed {SAMPLE}"},
            "e2e": {"value": round(value, 5), "unit": "draft blocks/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.cpu_probe:
        print(json.dumps(cpu_probe(args.cpu_probe)), flush=True)
        return
    rc = spawn_replicas(args)
    if rc is not None:
        sys.exit(rc)
    rank, ws = dist_setup()
    if args.impl == "reference":
        res = run_reference(args, rank, ws)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    res = run_ours(args, rank, ws)
    if rank == 0:
        if not args.no_cpu and ws == 1 and not args.profile_cycles:
            res["cpu_baseline"] = cpu_baseline()
            progress("CPU baseline")
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
