"""Benchmark: causal linear-attention tokens/s and fraction of the GB300 roofline.

A step is one causal forward + backward (la_forward then la_backward, the whole
training-direction hot path) over the B=4, H=8, N=16384, D=M=64 bf16 batch
resident in HBM. `value` is tokens/s over all ranks (a token is one sequence
position across all H heads). The JSON line also carries the forward-only,
non-causal and decode parts, the dominant kernel's roofline, the end-to-end
number through the C ABI with host buffers, and the fp64 oracle's CPU time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

import argparse
import json
import os
import shutil
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal linear-attention tokens/s (fwd, fwd+bwd, decode) and % of GB300 roofline"
MAIN = "causal_fwdbwd_b4h8n16384d64"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "source": "fallback"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    except Exception:
        return dict(FALLBACK_PEAKS)


# DRAM bytes per call measured with ncu (read + write, summed over the call's kernels) and the
# kernel-source revision they were taken on; reported only while the sources still match.
TRAFFIC_REVISION = "a3c3be67d9fcc426"
TRAFFIC_BYTES = {"la_backward": 902.3e6, "la_forward": 398.1e6}


def kernel_revision():
    import glob
    import hashlib
    files = sorted(glob.glob(os.path.join(ROOT, "kernelized_causal_self_gb300", "csrc", "*")))
    files.append(os.path.join(ROOT, "include", "la.h"))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# Algorithmic bytes per token-head (bf16 inputs, float32 gradients).
def fwd_bytes(w):
    return 2 * (2 * w.D + 2 * w.M)                     # q, k, v read + out written


def bwd_bytes(w):
    return 2 * (2 * w.D + 2 * w.M) + 4 * (2 * w.D + w.M)  # q,k,v,dout read; dq,dk,dv written


def decode_bytes(w):
    return 8 * w.D * w.M + 8 * w.D + 2 * (2 * w.D + 2 * w.M)  # S, Z read+write; q,k,v,out


EXTEND_TOKENS, EXTEND_POOL = 64, 512  # new tokens per stream per la_extend call; pool entries


def extend_bytes(w, T):
    """Per stream-head and call: q, k, v, out for T tokens + the state read and written."""
    return T * fwd_bytes(w) + 8 * w.D * w.M + 8 * w.D


def extend_setup(la, w, g, device, S, Z):
    """The decode workload's streams, their states scattered over a larger pool (stream b
    in entry 2b + 1), and EXTEND_TOKENS new tokens per stream."""
    import torch
    from kernelized_causal_self_gb300 import inputs
    T, P = EXTEND_TOKENS, EXTEND_POOL
    shp_qk, shp_v = (w.B, w.H, T, w.D), (w.B, w.H, T, w.M)
    eq = inputs.torch_normal(g, shp_qk, w.scale, w.dtype, device)
    ek = inputs.torch_normal(g, shp_qk, w.scale, w.dtype, device)
    ev = inputs.torch_normal(g, shp_v, w.scale, w.dtype, device)
    slots = ((2 * torch.arange(w.B, device=device) + 1) % P).to(torch.int32)
    pS = torch.zeros((P, w.H, w.D, w.M), dtype=torch.float32, device=device)
    pZ = torch.zeros((P, w.H, w.D), dtype=torch.float32, device=device)
    pS[slots.long()] = S
    pZ[slots.long()] = Z
    eo = torch.empty(shp_v, dtype=eq.dtype, device=device)
    ws = torch.empty(la.la_forward_workspace_bytes(w.B, w.H, T, w.D, w.M, True), dtype=torch.uint8,
                     device=device)
    return lambda: la.la_extend(eq, ek, ev, pS, pZ, slots=slots, out=eo, workspace=ws)


PACKED_MAX = 1024  # a serving batch: stream lengths uniform in 1..PACKED_MAX (seeded)


def packed_part(la, w, g, device, hbm, flush, reps, S, Z):
    """The decode workload's 256 streams (8 heads) continuing from their pool states
    with 1..PACKED_MAX new tokens each, in one la_extend_packed call on the packed
    token-major batch; beside it the same batch padded to its longest stream through
    la_extend with per-stream lengths."""
    import torch
    from kernelized_causal_self_gb300 import inputs
    P = EXTEND_POOL
    lens = inputs.stream_lengths(w.seed, w.B, 1, PACKED_MAX)
    cu = torch.zeros(w.B + 1, dtype=torch.int64)
    cu[1:] = torch.from_numpy(lens.astype("int64")).cumsum(0)
    T, N = int(cu[-1]), int(lens.max())
    cu = cu.to(torch.int32).to(device)
    pq = inputs.torch_normal(g, (T, w.H, w.D), w.scale, w.dtype, device)
    pk = inputs.torch_normal(g, (T, w.H, w.D), w.scale, w.dtype, device)
    pv = inputs.torch_normal(g, (T, w.H, w.M), w.scale, w.dtype, device)
    po = torch.empty((T, w.H, w.M), dtype=pq.dtype, device=device)
    slots = ((2 * torch.arange(w.B, device=device) + 1) % P).to(torch.int32)
    pS = torch.zeros((P, w.H, w.D, w.M), dtype=torch.float32, device=device)
    pZ = torch.zeros((P, w.H, w.D), dtype=torch.float32, device=device)
    pS[slots.long()] = S
    pZ[slots.long()] = Z
    ws = torch.empty(la.la_forward_workspace_bytes(w.B, w.H, N, w.D, w.M, True), dtype=torch.uint8,
                     device=device)
    ms = statistics.median(time_calls(
        lambda: la.la_extend_packed(pq, pk, pv, pS, pZ, cu, N, slots=slots, out=po, workspace=ws),
        reps, 3, flush))
    nbytes = T * w.H * fwd_bytes(w) + w.B * w.H * (8 * w.D * w.M + 8 * w.D)
    gbs = nbytes / (ms * 1e-3) / 1e9
    # the same streams padded to N tokens each
    dq = torch.zeros((w.B, w.H, N, w.D), dtype=pq.dtype, device=device)
    dk, dv = torch.zeros_like(dq), torch.zeros((w.B, w.H, N, w.M), dtype=pq.dtype, device=device)
    lt = torch.from_numpy(lens).to(device)
    for b in range(w.B):
        a, n = int(cu[b]), int(lens[b])
        for dst, src in ((dq, pq), (dk, pk), (dv, pv)):
            dst[b, :, :n] = src[a:a + n].transpose(0, 1)
    do = torch.empty_like(dv)
    del pq, pk, pv, po
    ms_pad = statistics.median(time_calls(
        lambda: la.la_extend(dq, dk, dv, pS, pZ, slots=slots, lens=lt, out=do, workspace=ws),
        reps, 3, flush))
    return {"tokens_per_s": T / (ms * 1e-3), "ms": ms, "tokens": T, "longest": N,
            "hbm_gbs": gbs, "roofline_frac": gbs / hbm, "padded_la_extend_ms": ms_pad,
            "lengths": f"uniform integers in 1..{PACKED_MAX}, seeded",
            "launch": "one la_extend_packed call", "l2": "flushed between calls (256 MB read)"}


class Clocks:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        exe = shutil.which("nvidia-smi")
        if exe is None:
            return self
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="la_clocks_", suffix=".csv")
        os.close(fd)
        self.proc = subprocess.Popen(
            [exe, "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
             "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.path is None:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def clock_index(device):
    """nvidia-smi index of `device` (its UUID), so the sampler watches the right GPU."""
    try:
        import torch
        return "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        return "0"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-parts", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the step's calls directly instead of replaying CUDA graphs")
    ap.add_argument("--part", default=None,
                    choices=["fwdbwd", "fwd16k", "fwd3072", "noncausal", "bwd", "bwdfwd", "decode",
                             "extend", "packed", "poly2", "rff"],
                    help="time one entry point on one workload only (for profilers)")
    return ap.parse_args()


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def device_inputs(w, device, dout=False):
    import torch
    from kernelized_causal_self_gb300 import inputs
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    q = inputs.torch_normal(g, (w.B, w.H, w.N, w.D), w.scale, w.dtype, device)
    k = inputs.torch_normal(g, (w.B, w.H, w.N, w.D), w.scale, w.dtype, device)
    v = inputs.torch_normal(g, (w.B, w.H, w.N, w.M), w.scale, w.dtype, device)
    if dout:
        d = inputs.torch_normal(g, (w.B, w.H, w.N, w.M), w.scale, w.dtype, device)
        return q, k, v, d, g
    return q, k, v, g


def l2_flush_buffer(device):
    """256 MB (twice the L2) read between timed calls to evict what the last call left."""
    import torch
    return torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device=device)


def flush_l2(buf):
    """Evict L2 by reading `buf` (a reduction, outside the timed region). A read leaves clean
    lines behind, so the next timed call pays no write-back of the flush's own lines, and the
    dirty lines of the previous call are written back here rather than inside the next one."""
    buf.sum()


def time_calls(fn, reps, warm, flush=None):
    """Per-call CUDA-event times (ms) on the current stream; optional L2 flush between calls."""
    import torch
    st = torch.cuda.current_stream()
    for _ in range(warm):
        fn()
    times = []
    for _ in range(reps):
        if flush is not None:
            flush_l2(flush)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        fn()
        b.record(st)
        b.synchronize()
        times.append(a.elapsed_time(b))
    return times


def run_parts(la, device, peaks, reps=10):
    """Forward-only, non-causal and decode throughput on their own workloads."""
    import torch
    from kernelized_causal_self_gb300 import inputs
    parts = {}
    flush = l2_flush_buffer(device)
    hbm = peaks["hbm_gbs"]
    for name in ("causal_fwdbwd_b4h8n16384d64", "causal_fwd_b8h8n3072d64",
                 "noncausal_fwd_b4h8n4096d64"):
        w = inputs.WORKLOADS[name]
        q, k, v, _ = device_inputs(w, device)
        out = torch.empty((w.B, w.H, w.N, w.M), dtype=q.dtype, device=device)
        ws = torch.empty(la.la_forward_workspace_bytes(w.B, w.H, w.N, w.D, w.M, w.causal),
                         dtype=torch.uint8, device=device)
        t = time_calls(lambda: la.la_forward(q, k, v, w.causal, out, ws), reps, 3, flush)
        ms = statistics.median(t)
        th = w.B * w.H * w.N
        gbs = th * fwd_bytes(w) / (ms * 1e-3) / 1e9
        key = ("causal_fwd_b4h8n16384d64" if name == MAIN else name)
        parts[key] = {"tokens_per_s": w.B * w.N / (ms * 1e-3), "ms": ms,
                      "hbm_gbs": gbs, "roofline_frac": gbs / hbm,
                      "l2": "flushed between calls (256 MB read)"}
        del q, k, v, out
    # decode: prefill, then the per-token steps replayed from a CUDA graph
    w = inputs.WORKLOADS["decode_s256h8d64_prefill1024_steps3072"]
    q, k, v, g = device_inputs(w, device)
    T = w.steps
    sq = inputs.torch_normal(g, (T, w.B, w.H, w.D), w.scale, w.dtype, device)
    sk = inputs.torch_normal(g, (T, w.B, w.H, w.D), w.scale, w.dtype, device)
    sv = inputs.torch_normal(g, (T, w.B, w.H, w.M), w.scale, w.dtype, device)
    outs = torch.empty((T, w.B, w.H, w.M), dtype=q.dtype, device=device)
    _, S, Z = la.la_prefill(q, k, v)
    S0, Z0 = S.clone(), Z.clone()
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for t in range(3):
            la.la_decode_step(sq[t], sk[t], sv[t], S, Z, out=outs[t])
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for t in range(T):
            la.la_decode_step(sq[t], sk[t], sv[t], S, Z, out=outs[t])

    def replay():
        S.copy_(S0)
        Z.copy_(Z0)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        b.synchronize()
        return a.elapsed_time(b)

    replay()
    ms = statistics.median([replay() for _ in range(3)])
    per_step = ms / T
    gbs = w.B * w.H * decode_bytes(w) / (per_step * 1e-3) / 1e9
    parts["decode_s256h8d64_prefill1024_steps3072"] = {
        "tokens_per_s": w.B * T / (ms * 1e-3), "ms_per_step": per_step, "hbm_gbs": gbs,
        "roofline_frac": gbs / hbm, "steps": T, "launch": "CUDA graph of 3072 la_decode_step calls",
        "l2": "S/Z state (33.5 MB) fits in L2; fraction can exceed 1"}
    # degree-2 polynomial feature map on the main workload's shape (forward, causal)
    parts["poly2_causal_fwd_b4h8n16384d64"] = poly2_part(la, inputs.WORKLOADS[MAIN], device, peaks,
                                                         flush, reps)
    # random Fourier features (F = 64) on the main workload's shape (forward, causal)
    parts["rff_causal_fwd_b4h8n16384d64"] = rff_part(la, inputs.WORKLOADS[MAIN], device, peaks,
                                                     flush, reps)
    # decode with a state too large for L2: DECODE_HBM_STREAMS streams x 8 heads (134 MB of S),
    # so every step reads and writes S in HBM
    parts[f"decode_s{DECODE_HBM_STREAMS}h{w.H}d{w.D}_hbm"] = decode_hbm_part(la, w, device, hbm)
    # extend: EXTEND_TOKENS new tokens per stream from states in a pool, one call
    fn = extend_setup(la, w, g, device, S0, Z0)
    ms = statistics.median(time_calls(fn, reps, 3, flush))
    gbs = w.B * w.H * extend_bytes(w, EXTEND_TOKENS) / (ms * 1e-3) / 1e9
    parts[f"extend_s256h8d64_t{EXTEND_TOKENS}_pool{EXTEND_POOL}"] = {
        "tokens_per_s": w.B * EXTEND_TOKENS / (ms * 1e-3), "ms": ms, "hbm_gbs": gbs,
        "roofline_frac": gbs / hbm, "same_tokens_as_decode_steps_ms": per_step * EXTEND_TOKENS,
        "launch": "one la_extend call", "l2": "flushed between calls (256 MB read)"}
    # the same streams as a packed serving batch of 1..PACKED_MAX new tokens each
    parts[f"extend_packed_s256h8d64_len1to{PACKED_MAX}_pool{EXTEND_POOL}"] = packed_part(
        la, w, g, device, hbm, flush, reps, S0, Z0)
    return parts


def poly2_flops(w):
    """Algorithmic flops per token-head of the degree-2 feature map (D^2 features): the
    read-out phi(q)^T S and the update S += phi(k) v^T, 2 D^2 M each (the intra-chunk
    products of the chunked form are implementation work, not counted)."""
    return 4 * w.D * w.D * w.M


def poly2_part(la, w, device, peaks, flush, reps):
    import torch
    q, k, v, _ = device_inputs(w, device)
    out = torch.empty_like(v)
    ws = torch.empty(la.la_poly2_workspace_bytes(w.B, w.H, w.N, w.D, w.M, True),
                     dtype=torch.uint8, device=device)
    ms = statistics.median(time_calls(lambda: la.la_forward_poly2(q, k, v, True, out, ws),
                                      reps, 3, flush))
    th = w.B * w.H * w.N
    tflops = th * poly2_flops(w) / (ms * 1e-3) / 1e12
    gbs = th * fwd_bytes(w) / (ms * 1e-3) / 1e9
    return {"tokens_per_s": w.B * w.N / (ms * 1e-3), "ms": ms, "tflops": tflops,
            "roofline_frac": tflops / peaks["bf16_tflops"], "bound": "tensor",
            "flops_per_token_head": poly2_flops(w), "hbm_gbs": gbs,
            "hbm_frac": gbs / peaks["hbm_gbs"], "l2": "flushed between calls (256 MB read)"}


RFF_FEATURES = 64


def rff_inputs(w, device):
    """W [F, D] with rows ~ N(0, I) (bf16) and phases b ~ U[0, 2 pi) (float32), seeded."""
    import torch
    from kernelized_causal_self_gb300 import inputs
    W = inputs.to_torch(inputs.normal(w.seed, (RFF_FEATURES, w.D), 1.0, w.dtype, 7), w.dtype, device)
    b = torch.from_numpy(inputs.uniform(w.seed, (RFF_FEATURES,), 0.0, 6.283185307179586, 8)).to(device)
    return W, b


def rff_part(la, w, device, peaks, flush, reps):
    """Causal forward with random Fourier features; HBM-bound like the elu + 1 forward (the
    feature GEMM is 2 * 2 * D * F flop per token-head), measured against the same 512 B per
    token-head (the features written and read back are implementation traffic)."""
    import torch
    q, k, v, _ = device_inputs(w, device)
    W, b = rff_inputs(w, device)
    out = torch.empty_like(v)
    ws = torch.empty(la.la_rff_workspace_bytes(w.B, w.H, w.N, w.D, w.M, RFF_FEATURES, True),
                     dtype=torch.uint8, device=device)
    ms = statistics.median(time_calls(lambda: la.la_forward_rff(q, k, v, W, b, True, out, ws),
                                      reps, 3, flush))
    th = w.B * w.H * w.N
    gbs = th * fwd_bytes(w) / (ms * 1e-3) / 1e9
    return {"tokens_per_s": w.B * w.N / (ms * 1e-3), "ms": ms, "hbm_gbs": gbs,
            "roofline_frac": gbs / peaks["hbm_gbs"], "bound": "hbm", "features": RFF_FEATURES,
            "l2": "flushed between calls (256 MB read)"}


DECODE_HBM_STREAMS, DECODE_HBM_STEPS, DECODE_HBM_PREFILL = 1024, 128, 128


def decode_hbm_part(la, w, device, hbm):
    """Decode steps over DECODE_HBM_STREAMS streams (the decode workload's heads, head size and
    inputs' distribution), whose float32 S/Z state (134 MB) exceeds the 129 MB L2: a prefill of
    DECODE_HBM_PREFILL tokens builds it, then a CUDA graph of DECODE_HBM_STEPS steps is timed."""
    import torch
    from kernelized_causal_self_gb300 import inputs
    n, T = DECODE_HBM_STREAMS, DECODE_HBM_STEPS
    g = torch.Generator(device=device)
    g.manual_seed(w.seed + 1)
    shp = (n, w.H, DECODE_HBM_PREFILL)
    q = inputs.torch_normal(g, shp + (w.D,), w.scale, w.dtype, device)
    k = inputs.torch_normal(g, shp + (w.D,), w.scale, w.dtype, device)
    v = inputs.torch_normal(g, shp + (w.M,), w.scale, w.dtype, device)
    _, S, Z = la.la_prefill(q, k, v)
    del q, k, v
    sq = inputs.torch_normal(g, (T, n, w.H, w.D), w.scale, w.dtype, device)
    sk = inputs.torch_normal(g, (T, n, w.H, w.D), w.scale, w.dtype, device)
    sv = inputs.torch_normal(g, (T, n, w.H, w.M), w.scale, w.dtype, device)
    outs = torch.empty((T, n, w.H, w.M), dtype=sq.dtype, device=device)
    S0, Z0 = S.clone(), Z.clone()
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for t in range(3):
            la.la_decode_step(sq[t], sk[t], sv[t], S, Z, out=outs[t])
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for t in range(T):
            la.la_decode_step(sq[t], sk[t], sv[t], S, Z, out=outs[t])

    def replay():
        S.copy_(S0)
        Z.copy_(Z0)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        b.synchronize()
        return a.elapsed_time(b)

    replay()
    ms = statistics.median([replay() for _ in range(3)])
    per_step = ms / T
    gbs = n * w.H * decode_bytes(w) / (per_step * 1e-3) / 1e9
    return {"tokens_per_s": n * T / (ms * 1e-3), "ms_per_step": per_step, "hbm_gbs": gbs,
            "roofline_frac": gbs / hbm, "steps": T, "streams": n,
            "launch": f"CUDA graph of {T} la_decode_step calls",
            "l2": f"S/Z state ({n * w.H * (w.D * w.M + w.D) * 4 / 1e6:.0f} MB) exceeds L2: "
                  "an HBM-bound step"}


def run_ours(args, world, rank, local):
    import torch
    import kernelized_causal_self_gb300 as la
    from kernelized_causal_self_gb300 import build as labuild
    from kernelized_causal_self_gb300 import inputs

    labuild.build()
    la.load_library()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    peaks = load_peaks()
    w = inputs.WORKLOADS[MAIN]
    q, k, v, dout, _ = device_inputs(w, device, dout=True)
    out = torch.empty((w.B, w.H, w.N, w.M), dtype=q.dtype, device=device)
    f32 = torch.float32
    dq = torch.empty((w.B, w.H, w.N, w.D), dtype=f32, device=device)
    dk = torch.empty((w.B, w.H, w.N, w.D), dtype=f32, device=device)
    dv = torch.empty((w.B, w.H, w.N, w.M), dtype=f32, device=device)
    wsf = torch.empty(la.la_forward_workspace_bytes(w.B, w.H, w.N, w.D, w.M, True),
                      dtype=torch.uint8, device=device)
    wsb = torch.empty(la.la_backward_workspace_bytes(w.B, w.H, w.N, w.D, w.M, True),
                      dtype=torch.uint8, device=device)
    st = torch.cuda.current_stream(device)
    K, W = args.steps, args.warmup
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]

    def fwd():
        la.la_forward(q, k, v, True, out, wsf)

    def bwd():  # the training order: the backward reads the forward's segment states
        la.la_backward(q, k, v, dout, True, dq, dk, dv, wsb, fwd_workspace=wsf)

    # Each call is captured once into a CUDA graph (kernels + workspace memsets,
    # with programmatic-dependent-launch edges) and replayed per step.
    per_step_launches = None
    if not args.no_graph:
        side = torch.cuda.Stream(device)
        side.wait_stream(st)
        with torch.cuda.stream(side):
            for _ in range(2):
                fwd()
                bwd()
        st.wait_stream(side)
        torch.cuda.synchronize()
        graphs = []
        per_step_launches = 0
        for fn in (fwd, bwd):
            gph = torch.cuda.CUDAGraph()
            c0 = la.la_kernel_launches()
            with torch.cuda.graph(gph):
                fn()
            per_step_launches += la.la_kernel_launches() - c0
            graphs.append(gph)
        fwd_run, bwd_run = graphs[0].replay, graphs[1].replay
    else:
        fwd_run, bwd_run = fwd, bwd

    def step(i=None):
        if i is not None:
            ev[i][0].record(st)
        fwd_run()
        if i is not None:
            ev[i][1].record(st)
        bwd_run()
        if i is not None:
            ev[i][2].record(st)

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    barrier(world)
    n0 = la.la_kernel_launches()
    with Clocks(clock_index(device)) as clk:
        torch.cuda.synchronize()
        barrier(world)
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(st)
        for i in range(K):
            step(i)
        t_end.record(st)
        torch.cuda.synchronize()
        barrier(world)
    launches = la.la_kernel_launches() - n0
    if per_step_launches is not None:   # graph replays launch what was captured
        launches = per_step_launches * K
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), world, device)
    ms_step = ms_total / K
    tokens = w.B * w.N * world
    value = tokens / (ms_step * 1e-3)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    th = w.B * w.H * w.N
    hbm = peaks["hbm_gbs"]
    cand = {"la_backward": (bwd_ms, th * bwd_bytes(w), bwd_bytes(w)),
            "la_forward": (fwd_ms, th * fwd_bytes(w), fwd_bytes(w))}
    dom = max(cand, key=lambda n: cand[n][0])
    d_ms, d_bytes, per_unit = cand[dom]
    achieved = d_bytes / (d_ms * 1e-3) / 1e9
    rev = kernel_revision()
    traffic = TRAFFIC_BYTES.get(dom) if rev == TRAFFIC_REVISION else None
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic, "kernel_revision": rev,
                "peak_source": peaks.get("source"),
                "algorithmic_bytes_per_token_head": per_unit, "token_heads_per_launch": th,
                "launch_ms": d_ms, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms}

    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": MAIN, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "M": w.M,
                   "step": "la_forward + la_backward (causal; the backward reads the "
                           "forward's segment states from its workspace)", "grads": "float32",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "launch": "CUDA graph replay per call" if per_step_launches is not None
                   else "direct launches",
                   "l2": "inputs+outputs 470 MB per step > 129 MB L2 (no flush needed)"},
        "roofline": roofline, "gpu_launches": int(launches),
        "clocks": clk.summary(),
    }
    if not args.no_e2e:
        result["e2e"] = run_e2e(la, w, q, k, v, dout, device, K=max(2, min(K, 5)))
    if not args.no_parts:
        del q, k, v, dout, dq, dk, dv, out
        torch.cuda.empty_cache()
        result["parts"] = run_parts(la, device, peaks)
    if rank == 0 and world == 1 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(result), flush=True)


def run_e2e(la, w, q, k, v, dout, device, K):
    """Same step through the C ABI with pinned host buffers, host <-> device copies inside
    the timed region. The step is cut into its B batch slices (independent sequences) and
    pipelined over three streams: copy-in (H2D of q, k, v, dout), compute (la_forward +
    la_backward per slice) and copy-out (D2H of out, dq, dk, dv), so the two copy directions
    and the kernels overlap, within a step and across consecutive steps."""
    import torch
    f32 = torch.float32
    hq, hk, hv, hd = (t.cpu().pin_memory() for t in (q, k, v, dout))
    ho = torch.empty(tuple(q.shape[:3]) + (w.M,), dtype=q.dtype).pin_memory()
    hdq = torch.empty(q.shape, dtype=f32).pin_memory()
    hdk = torch.empty(q.shape, dtype=f32).pin_memory()
    hdv = torch.empty(tuple(q.shape[:3]) + (w.M,), dtype=f32).pin_memory()
    o = torch.empty(ho.shape, dtype=q.dtype, device=device)
    gq = torch.empty(q.shape, dtype=f32, device=device)
    gk = torch.empty(q.shape, dtype=f32, device=device)
    gv = torch.empty(hdv.shape, dtype=f32, device=device)
    dt = la.LA_BF16 if q.dtype == torch.bfloat16 else la.LA_F32
    wf = torch.empty((la.la_forward_workspace_bytes(1, w.H, w.N, w.D, w.M, True, dt),),
                     dtype=torch.uint8, device=device)
    wb = torch.empty((la.la_backward_workspace_bytes(1, w.H, w.N, w.D, w.M, True, dt),),
                     dtype=torch.uint8, device=device)
    s_in, s_cmp, s_out = (torch.cuda.Stream(device=device) for _ in range(3))
    nb = w.B
    e_in = [torch.cuda.Event() for _ in range(nb)]
    e_done = [torch.cuda.Event() for _ in range(nb)]
    e_out = [torch.cuda.Event() for _ in range(nb)]

    def step():
        for b in range(nb):  # inputs of slice b, once the previous step's compute is done with them
            s_in.wait_event(e_done[b])
            with torch.cuda.stream(s_in):
                for dst, src in ((q, hq), (k, hk), (v, hv), (dout, hd)):
                    dst[b].copy_(src[b], non_blocking=True)
                e_in[b].record(s_in)
        for b in range(nb):  # compute, once the inputs are in and last step's outputs are out
            s_cmp.wait_event(e_in[b])
            s_cmp.wait_event(e_out[b])
            with torch.cuda.stream(s_cmp):
                sl = slice(b, b + 1)
                la.la_forward(q[sl], k[sl], v[sl], True, out=o[sl], workspace=wf)
                la.la_backward(q[sl], k[sl], v[sl], dout[sl], True, dq=gq[sl], dk=gk[sl], dv=gv[sl],
                               workspace=wb, fwd_workspace=wf)
                e_done[b].record(s_cmp)
        for b in range(nb):
            s_out.wait_event(e_done[b])
            with torch.cuda.stream(s_out):
                for dst, src in ((ho, o), (hdq, gq), (hdk, gk), (hdv, gv)):
                    dst[b].copy_(src[b], non_blocking=True)
                e_out[b].record(s_out)

    cur = torch.cuda.current_stream(device)
    step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    a.record(cur)
    for st in (s_in, s_cmp, s_out):
        st.wait_event(a)
    for _ in range(K):
        step()
    cur.wait_event(e_out[nb - 1])  # the last copy-out depends on every earlier operation
    z.record(cur)
    z.synchronize()
    ms = a.elapsed_time(z) / K
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hd))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hdq, hdk, hdv))
    return {"value": w.B * w.N / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "path": f"pinned host -> device, la_forward + la_backward, device -> pinned host; "
                    f"{nb} batch slices pipelined over copy-in, compute and copy-out streams"}


def _oracle_worker_init():
    """Pool worker set-up: one BLAS/OpenMP thread per process (the pool supplies the cores)."""
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    import oracle  # noqa: F401  (import cost kept out of the timed map)


def _oracle_fwdbwd(task):
    """Causal forward + backward of one (b, h) sequence of `n` positions with the fp64 oracle,
    as it stands; the inputs are drawn like the workload's (seed, sample index)."""
    seed, idx, n, D, M, scale, dtype = task
    import oracle
    from kernelized_causal_self_gb300 import inputs
    q, k, v = inputs.qkv(seed * 100003 + idx, 1, 1, n, D, M, scale, dtype)
    g = inputs.upstream_grad(seed * 100003 + idx, 1, 1, n, M, scale, dtype)
    q, k, v, g = q[0, 0], k[0, 0], v[0, 0], g[0, 0]
    t0 = time.perf_counter()
    oracle.forward(q, k, v, True)
    oracle.backward(q, k, v, g, True)
    return time.perf_counter() - t0


class OraclePool:
    """The fp64 oracle on the host's cores: one worker process per core, started with `spawn`
    (safe after CUDA has been initialised), each running whole (b, h) sequences."""

    def __init__(self, cores=None):
        import multiprocessing as mp
        self.cores = int(cores or os.cpu_count() or 1)
        self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_oracle_worker_init)

    def run(self, w, n, n_seq, offset=0):
        """Wall time (s) of n_seq sequences of n positions spread over the workers."""
        tasks = [(w.seed, offset + i, n, w.D, w.M, w.scale, w.dtype) for i in range(n_seq)]
        t0 = time.perf_counter()
        self.pool.map(_oracle_fwdbwd, tasks, chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(w):
    """fp64 oracle (as it stands) on the host's cores: causal forward + backward of whole (b, h)
    sequences of the workload, one sequence per core, timed after a warm-up round."""
    pool = OraclePool()
    try:
        pool.run(w, 256, pool.cores)                  # workers up, imports done
        sec = pool.run(w, w.N, pool.cores, offset=1000)
    finally:
        pool.close()
    tokens = pool.cores * w.N / w.H   # one head of N positions = N/H token-equivalents
    return {"value": tokens / sec, "unit": "tokens/s", "cores": pool.cores,
            "host_cpus": os.cpu_count(), "kind": "oracle",
            "sample": f"{pool.cores} (b,h) sequences of N={w.N} (one per core, {pool.cores} worker "
                      f"processes), causal fwd + bwd, float64 NumPy recurrence, {sec:.1f} s wall"}


def run_reference(args, world, rank):
    """Reference arm: the fp64 oracle on the host's cores, a bounded sample per step."""
    if rank != 0:
        return
    from kernelized_causal_self_gb300 import inputs
    w = inputs.WORKLOADS[MAIN]
    n = 2048   # first 2048 positions of one (b, h) sequence per core per step
    pool = OraclePool()
    try:
        for i in range(args.warmup):
            pool.run(w, n, pool.cores, offset=i * pool.cores)
        secs = [pool.run(w, n, pool.cores, offset=(args.warmup + i) * pool.cores)
                for i in range(args.steps)]
    finally:
        pool.close()
    sec = sum(secs) / len(secs)
    value = pool.cores * (n / w.H) / sec
    sample = (f"per step: causal fwd + bwd of {n} positions of {pool.cores} (b,h) sequences of "
              f"{MAIN} (one per core, {pool.cores} worker processes), float64 NumPy oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": MAIN, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "M": w.M,
                   "sample_positions": n, "sequences_per_step": pool.cores},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": pool.cores, "kind": "oracle",
                         "host_cpus": os.cpu_count(), "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_part(args):
    """One entry point on one workload, W + K calls; prints per-call CUDA-event times."""
    import torch
    import kernelized_causal_self_gb300 as la
    from kernelized_causal_self_gb300 import build as labuild
    from kernelized_causal_self_gb300 import inputs
    labuild.build()
    la.load_library()
    device = torch.device("cuda", 0)
    name = {"fwdbwd": MAIN, "fwd16k": MAIN, "bwd": MAIN, "bwdfwd": MAIN, "poly2": MAIN, "rff": MAIN,
            "fwd3072": "causal_fwd_b8h8n3072d64",
            "noncausal": "noncausal_fwd_b4h8n4096d64",
            "decode": "decode_s256h8d64_prefill1024_steps3072",
            "extend": "decode_s256h8d64_prefill1024_steps3072",
            "packed": "decode_s256h8d64_prefill1024_steps3072"}[args.part]
    w = inputs.WORKLOADS[name]
    q, k, v, dout, g = device_inputs(w, device, dout=True)
    if args.part == "decode":
        _, S, Z = la.la_prefill(q, k, v)
        sq = inputs.torch_normal(g, (w.B, w.H, w.D), w.scale, w.dtype, device)
        sk = inputs.torch_normal(g, (w.B, w.H, w.D), w.scale, w.dtype, device)
        sv = inputs.torch_normal(g, (w.B, w.H, w.M), w.scale, w.dtype, device)
        fn = lambda: la.la_decode_step(sq, sk, sv, S, Z)
    elif args.part == "extend":
        _, S, Z = la.la_prefill(q, k, v)
        fn = extend_setup(la, w, g, device, S, Z)
    elif args.part == "packed":  # times both calls itself: prints its parts entry
        _, S, Z = la.la_prefill(q, k, v)
        entry = packed_part(la, w, g, device, load_peaks()["hbm_gbs"], l2_flush_buffer(device),
                            max(args.steps, 1), S, Z)
        print(json.dumps({"part": args.part, "workload": name, **entry}), flush=True)
        return
    elif args.part == "bwd":
        fn = lambda: la.la_backward(q, k, v, dout, True)
    elif args.part == "bwdfwd":  # the backward reading a forward's segment states
        wsf = torch.empty(la.la_forward_workspace_bytes(w.B, w.H, w.N, w.D, w.M, True),
                          dtype=torch.uint8, device=device)
        la.la_forward(q, k, v, True, workspace=wsf)
        fn = lambda: la.la_backward(q, k, v, dout, True, fwd_workspace=wsf)
    elif args.part == "poly2":
        fn = lambda: la.la_forward_poly2(q, k, v, True)
    elif args.part == "rff":
        W, b = rff_inputs(w, device)
        fn = lambda: la.la_forward_rff(q, k, v, W, b, True)
    elif args.part == "fwdbwd":
        fn = lambda: (la.la_forward(q, k, v, True), la.la_backward(q, k, v, dout, True))
    else:
        fn = lambda: la.la_forward(q, k, v, w.causal)
    t = time_calls(fn, args.steps, args.warmup)
    print(json.dumps({"part": args.part, "workload": name, "ms": t,
                      "median_ms": statistics.median(t)}), flush=True)


def _free_port():
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_replicas(n, argv, script=None):
    """Run `script` (this file by default) as n local processes, one per GPU: rank r gets
    RANK = LOCAL_RANK = r, WORLD_SIZE = n and a 127.0.0.1 rendezvous, as torchrun would set
    them. The replicas share nothing on the data path; they meet only at the barriers around
    the timed region and in the max over ranks. Returns the worst exit code."""
    port = str(_free_port())
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=port)
        procs.append(subprocess.Popen([sys.executable, script or os.path.abspath(__file__), *argv],
                                      env=env))
    codes = [p.wait() for p in procs]
    return max(codes, key=abs)


def main():
    args = parse()
    if args.part is not None:
        run_part(args)
        return
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # not started by torchrun: start the replicas here, one process per GPU
        if args.impl == "ours":
            import torch
            if torch.cuda.device_count() < args.gpus:
                sys.exit(f"bench.py --gpus {args.gpus}: only {torch.cuda.device_count()} CUDA "
                         "device(s) visible")
        sys.exit(launch_replicas(args.gpus, sys.argv[1:]))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup(args)
    run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
