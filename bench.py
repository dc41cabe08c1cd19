"""Benchmark of the GB300 ZeRO-DP optimizer step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--config 1..5] [--nd N] [--qgather] [--qgz] [--accum K]
                    [--offload] [--serial] [--gathers 1|2] [--row-pad N]
                    [--param-dtype bf16|fp16] [--stage 1|2]
                    [--psi N] [--no-cpu-baseline] [--no-e2e]

A step is one pass of the whole hot path (reduce-scatter of the simulated
ranks' gradients, global checks, Adam on every shard, 16-bit cast and gather)
over one batch of synthetic gradients already resident in HBM.  The default
workload is the largest that fits one GPU: the ZeRO-3 layer-wise step over 8
Llama-3-8B-shaped decoder layers (Psi_l = 218,112,000 each), N_d = 16
simulated ranks, bf16 gradients ~N(0, 1e-3), Adam lr 1e-3; per layer the
all-gather of its bf16 shards, then the reduce-scatter of its ranks'
gradients, Adam and the bf16 shards, through one call of the layer loop
(the next layer's gather on a second stream).  --config 2 is the GPT-2-small
clipped ZeRO-2 step, --config 3 the GPT-2 1.5B fp16 loss-scaled step,
--config 5 the N_d sweep at Psi = 2^28, --config 1 the small parity case.

One JSON line is printed (rank 0).  value = parameters updated per second over
the whole job; roofline = the dominant kernel's algorithmic bytes per launch
over its CUDA-event duration, against the measured HBM copy bandwidth;
cpu_baseline = the CPU oracle timed on a bounded sample on this host;
e2e = the same metric with the gradients copied from pinned host memory and
the updated 16-bit parameters copied back inside the timed region.

--gpus N under torchrun runs N independent replicas (one per GPU): the
ranks of the method are buffers inside one GPU, so nothing is exchanged
between GPUs; the timed region is bracketed by barriers and the max over
ranks is taken.  --impl reference times the CPU oracle instead.
"""
import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ZeRO step params/s and achieved HBM GB/s (% of GB300 roofline), 1 GPU"
UNIT = "params/s"
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------- workloads
def workload(cfg, nd=None, qgather=False, psi=None, qgz=False, gathers=1, offload=False, accum=1, serial=False,
             param_dtype=None, stage=None):
    """Sizes, hyper-parameters and the algorithmic bytes of one step.  psi
    overrides the parameter count (a smaller case of the same workload, for
    profiling).  serial: the ZeRO-3 layer loop with every gather on the step's
    stream (default: the gathers on a second stream, the next layer's
    overlapping this layer's step).  param_dtype ("bf16"/"fp16"): the 16-bit
    parameter dtype (default bf16; the fp16-gradient workload pairs fp16
    parameters with fp16 gradients when asked).  stage: 1 or 2 for the ZeRO-1/2
    workloads (the same math; the label and the plan's stage)."""
    args = dict(cfg=cfg, nd=nd, qgather=qgather, psi=psi, qgz=qgz, gathers=gathers, offload=offload, accum=accum,
                serial=serial, param_dtype=param_dtype, stage=stage)
    if cfg == 1:
        w = dict(name="zero2_psi1000003_nd4_adam", psi=1_000_003, n_d=4, stage=2, pad=8, gdt="bf16",
                 sigma=1e-3, tail=False, lr=1e-3, b2=0.999, wd=0.0, clip=0.0, ls=False, layers=1)
    elif cfg == 2:
        w = dict(name="zero2_gpt2small_psi124439808_nd8_adamw_clip1", psi=124_439_808, n_d=8, stage=2, pad=8,
                 gdt="bf16", sigma=1e-2, tail=True, lr=3e-4, b2=0.95, wd=0.1, clip=1.0, ls=False, layers=1)
    elif cfg == 3:
        w = dict(name="zero2_gpt2xl_psi1500000000_nd8_fp16_lossscale", psi=1_500_000_000, n_d=8, stage=2, pad=8,
                 gdt="fp16", sigma=1e-4, tail=False, lr=1e-4, b2=0.999, wd=0.0, clip=0.0, ls=True, layers=1)
    elif cfg == 4:
        # gathers: per layer and step, 1 (the workload as configured) or 2
        # (forward and backward, the pages' 3-psi communication volume)
        w = dict(name="zero3_llama3_8b_8layers_psil218112000_nd16" + ("_2gathers" if gathers == 2 else ""),
                 psi=218_112_000, n_d=16, stage=3, pad=8, gdt="bf16", sigma=1e-3, tail=False, lr=1e-3, b2=0.999,
                 wd=0.0, clip=0.0, ls=False, layers=8, gathers=gathers)
    elif cfg == 5:
        n = nd or 8
        w = dict(name="zero2_psi2p28_nd%d" % n, psi=1 << 28, n_d=n, stage=2, pad=8, gdt="bf16", sigma=1e-3,
                 tail=False, lr=1e-3, b2=0.999, wd=0.0, clip=0.0, ls=False, layers=1)
    else:
        raise SystemExit("unknown config %r" % cfg)
    if qgather and not qgz and w["stage"] == 3:
        # the ZeRO-3 layer loop with block-int8 quantized gathers (qwZ): each
        # layer's gather writes int8 codes, block scales and the dequantized
        # bf16 values instead of the bf16 shards
        w["qgather"] = True
        w["name"] += "_qgather"
    elif qgather or qgz:
        # the ZeRO++ variants of the bf16 ZeRO-2 workloads: the int8 gather
        # epilogue, int8 codes + block scales as the ranks' gradients, or both
        if w["stage"] == 3 or w["gdt"] != "bf16":
            raise SystemExit("--qgather applies to the bf16 workloads (configs 1, 2, 4, 5), --qgz to the bf16 "
                             "ZeRO-2 ones (configs 1, 2, 5)")
        w["qgather"], w["qgz"] = qgather, qgz
        w["name"] += ("_qgz" if qgz else "") + ("_qgather" if qgather else "")
        if qgz:
            w["pad"] = 16     # int8 shard slices start 16-byte aligned
    if psi:
        w["psi"] = int(psi)
        w["name"] += "_psi%d" % w["psi"]
    if offload:
        # optimizer state in page-locked host memory, read and written over the CPU-GPU link
        w["offload"] = True
        w["name"] += "_offload"
    if w["stage"] == 3:
        # the next layer's gather on a second stream while this layer's step runs
        # (the layer loop's overlap), unless asked to keep one stream
        w["overlap"] = not serial
        if serial:
            w["name"] += "_serial"
    elif serial:
        raise SystemExit("--serial applies to the ZeRO-3 layer loop (config 4)")
    w["pdt"] = "bf16"
    if param_dtype:
        if w.get("qgather") and param_dtype != "bf16":
            raise SystemExit("the int8 gather takes bf16 parameters")
        w["pdt"] = param_dtype
        w["name"] += "_params_" + param_dtype
    if stage:
        if w["stage"] == 3 or stage not in (1, 2):
            raise SystemExit("--stage 1|2 applies to the ZeRO-1/2 workloads (configs 1, 2, 3, 5)")
        if stage != w["stage"]:
            w["stage"] = stage
            w["name"] = ("zero%d" % stage) + w["name"][5:]
    if accum > 1:
        if w["stage"] == 3 or w.get("qgz") or w.get("qgather") or offload or w["ls"]:
            raise SystemExit("--accum applies to the plain and clipped ZeRO-2 workloads (configs 1, 2, 5)")
        w["accum"] = accum
        w["name"] += "_accum%d" % accum
    n_d = w["n_d"]
    # algorithmic bytes per parameter of one step (minimum HBM traffic)
    if w.get("accum"):
        # micro-batch 1 writes the fp32 accumulator, 2..k-1 read and write it,
        # the step at micro-batch k reads it in each pass that reads the ranks
        k = w["accum"]
        micro = (2 * n_d + 4) + (k - 2) * (2 * n_d + 8)
        if w["clip"] > 0:
            final = 2 * n_d + 38 if n_d > 4 else 4 * n_d + 34
        else:
            final = 2 * n_d + 30
        w["bytes_per_param"] = micro + final
    elif w.get("qgz") and w.get("qgather"):
        # int8 codes in, int8 gather out; clipped, a reduce pass over the codes
        # first: for n_d > 4 it writes the fp32 reduced gradient, which the
        # Adam pass with the int8 gather reads, else the update re-reads the codes
        q = n_d * (1 + 4.0 / 2048)
        if w["clip"] > 0 and n_d > 4:
            w["bytes_per_param"] = (q + 4) + (4 + 27 + 4.0 / 2048)
        else:
            w["bytes_per_param"] = q + 27 + 4.0 / 2048 + (q if w["clip"] > 0 else 0)
    elif w.get("qgz"):
        # the receiver reads int8 codes + one fp32 scale per 2048 per rank;
        # clipped, the reduce pass over them comes first, writing the fp32
        # reduced gradient for the Adam pass when n_d > 4
        q = n_d * (1 + 4.0 / 2048)
        if w["clip"] > 0:
            w["bytes_per_param"] = q + 34 if n_d > 4 else 2 * q + 26
        else:
            w["bytes_per_param"] = q + 26
    elif w["stage"] == 3:
        # per gather: the 16-bit shards read and the gathered values written,
        # or with qwZ the shards read, codes + block scales + dequantized bf16 written
        per_gather = (5 + 4.0 / 2048) if w.get("qgather") else 4
        w["bytes_per_param"] = 2 * n_d + 26 + per_gather * w.get("gathers", 1)
    elif w.get("qgather"):
        # clipped: for n_d > 4 the reduce pass writes the fp32 reduced gradient
        # and the Adam pass with the int8 gather reads it; else a read-only
        # reduce pass, then the fused step re-reads the ranks
        if w["clip"] > 0 and n_d > 4:
            w["bytes_per_param"] = (2 * n_d + 4) + (4 + 27 + 4.0 / 2048)
        else:
            w["bytes_per_param"] = 2 * n_d + 27 + 4.0 / 2048 + (2 * n_d if w["clip"] > 0 else 0)
    elif w["clip"] > 0:
        w["bytes_per_param"] = 2 * n_d + 34 if n_d > 4 else 4 * n_d + 26
    else:
        w["bytes_per_param"] = 2 * n_d + 26
    w["psi_total"] = w["psi"] * w["layers"]
    w["args"] = args
    return w


def workload_from_args(args):
    w = workload(args.config, args.nd, args.qgather, args.psi, args.qgz, args.gathers, args.offload, args.accum,
                 args.serial, args.param_dtype, args.stage)
    if args.row_pad:
        w["row_pad"] = args.row_pad
        w["name"] += "_rowpad%d" % args.row_pad
    return w


def config_of(w, world):
    """The JSON line's config: the workload by name and size (both arms print
    the same)."""
    small = w["psi_total"] * w["bytes_per_param"] < 4 * L2_BYTES
    c = {"workload": w["name"], "psi": w["psi"], "layers": w["layers"], "n_d": w["n_d"], "stage": w["stage"],
         "grad_dtype": w["gdt"], "param_dtype": w["pdt"], "clip": w["clip"], "loss_scaling": w["ls"],
         "bytes_per_param": w["bytes_per_param"], "micro_batches": w.get("accum", 1),
         "rank_row_pad": w.get("row_pad", 0), "parallelism": "replicas x%d" % world,
         "l2": "flushed between steps" if small else "inputs larger than L2"}
    if w["stage"] == 3:
        c["gathers_per_layer"] = w.get("gathers", 1)
        c["gather_stream"] = "second stream, overlapping the steps" if w.get("overlap") else "the step's stream"
    return c


# ------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons, keeping the samples taken while
    the timed region ran (mark() brackets it)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []          # (arrival time, line)
        self.window = [None, None]

    def mark(self, which):
        self.window[which] = time.monotonic()

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = self.window
        inside = [ln for t, ln in self.lines if t0 is not None and t1 is not None and t0 <= t <= t1 + 0.05]
        if not inside and self.lines:
            # a timed region shorter than the sampling period: the sample nearest to it
            mid = (t0 + t1) / 2 if t0 is not None and t1 is not None else self.lines[-1][0]
            inside = [min(self.lines, key=lambda x: abs(x[0] - mid))[1]]
        for ln in inside:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for k, n in enumerate(names):
                if f[5 + k].lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples_in_timed_region": len(sm)}


# ---------------------------------------------------------------- GPU arm
def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# nominal HBM3e bandwidth of the part: a second denominator for the step's
# fraction, beside the measured copy bandwidth that the roofline uses
NOMINAL_HBM_GBS = 8000.0


# ncu DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum), per
# kernel and workload, with a hash of the kernel sources they were taken on;
# reported as null once the sources change.
TRAFFIC = {
    # one-pass full-size captures (dram__bytes_read.sum + dram__bytes_write.sum):
    # the per-layer fused step of the 8-layer workload, 9.597 GB read + 3.020 GB
    # written (two launches' mean); the GPT-2-small clipped step's Adam pass,
    # 1.991 + 1.680 GB
    ("fused_step", "zero3_llama3_8b_8layers_psil218112000_nd16"): {"bytes": 12.617e9, "src": "89dae4f5ae82"},
    ("adam_shard", "zero2_gpt2small_psi124439808_nd8_adamw_clip1"): {"bytes": 3.671e9, "src": "89dae4f5ae82"},
}


def _code_only(text):
    """C++ source without its comments and with its whitespace collapsed (the
    engine's sources hold no string literal containing a comment marker)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash():
    """Hash of the streaming engine's device code and of its argument block
    (the StreamArgs definition), comments and layout left out: the kernels
    whose traffic TRAFFIC records.  Host-only changes elsewhere, and edits
    of comments, leave those kernels, and their traffic, as they were."""
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "zero_optimizer_step_02_gb300", "csrc")
    for f in ("zk_stream.cu", "zk_common.cuh"):
        with open(os.path.join(csrc, f)) as fh:
            h.update(_code_only(fh.read()).encode())
    with open(os.path.join(csrc, "zk_launch.h")) as fh:
        text = fh.read()
    a = text.index("struct StreamArgs {")
    h.update(_code_only(text[a:text.index("};", a)]).encode())
    return h.hexdigest()[:12]


class Job:
    """Device buffers of one replica's workload."""

    def __init__(self, w, device, pool=2):
        import torch
        import zero_optimizer_step_02_gb300 as z
        from zero_optimizer_step_02_gb300 import synth
        self.z, self.torch, self.w = z, torch, w
        gdt = z.ZERO_FP16 if w["gdt"] == "fp16" else z.ZERO_BF16
        pdt = z.ZERO_FP16 if w["pdt"] == "fp16" else z.ZERO_BF16
        self.hp = z.hparams(lr=w["lr"], beta1=0.9, beta2=w["b2"], eps=1e-8, weight_decay=w["wd"],
                            max_norm=w["clip"], loss_scaling=w["ls"])
        self.plan = z.Plan(w["psi"], w["n_d"], stage=w["stage"], grad_dtype=gdt, shard_pad=w["pad"],
                           param_dtype=pdt)
        lp_dt = torch.float16 if pdt == z.ZERO_FP16 else torch.bfloat16
        tdt = torch.float16 if gdt == z.ZERO_FP16 else torch.bfloat16
        row = z.row_len(w["psi"], w.get("row_pad", 0))
        scale = 1024.0 if w["ls"] else 1.0
        # gradient sets: one per layer for ZeRO-3, else a small pool used in turn
        nsets = w["layers"] if w["layers"] > 1 else pool
        self.grads = []
        for k in range(nsets):
            g = torch.empty(w["n_d"], row, dtype=tdt, device=device)
            for r in range(w["n_d"]):
                synth.gaussian_(g[r, :w["psi"]], w["sigma"], 20261202 + k, r, heavy_tail=w["tail"], scale=scale)
            self.grads.append(g)
        L = w["layers"]
        n = self.plan.padded
        self.master = [synth.master_init(n, w["psi"], 7 + l, device=device) for l in range(L)]
        self.m = [torch.zeros(n, device=device) for _ in range(L)]
        self.v = [torch.zeros(n, device=device) for _ in range(L)]
        self.offload = w.get("offload", False)
        if self.offload:
            self.master = [x.cpu().pin_memory() for x in self.master]
            self.m = [torch.zeros(n).pin_memory() for _ in range(L)]
            self.v = [torch.zeros(n).pin_memory() for _ in range(L)]
        self.pingpong = w["ls"]
        if self.pingpong:
            self.master2 = [torch.zeros(n, device=device) for _ in range(L)]
            self.m2 = [torch.zeros(n, device=device) for _ in range(L)]
            self.v2 = [torch.zeros(n, device=device) for _ in range(L)]
        lp_n = n if w["stage"] == 3 else w["psi"]
        self.lp = [torch.zeros(lp_n, dtype=lp_dt, device=device) for _ in range(L)]
        if w["stage"] == 3:
            # the ZeRO-3 layer loop: two gathered buffers used in turn (layer l
            # into buffer l % 2), the gathers on a second stream unless serial
            self.gathered = [torch.zeros(w["psi"], dtype=lp_dt, device=device) for _ in range(2)]
            self.gather_stream = torch.cuda.Stream(device=device) if w.get("overlap") else None
            self.stack = z.LayerStack([(self.plan.handle, self.ranks(l), self.master[l], self.m[l], self.v[l],
                                        self.lp[l]) for l in range(L)])
        self.gq_codes_l = self.gq_scales_l = None
        if w.get("qgather"):
            nbs = -(-self.plan.shard // 2048)
            self.gq_codes = torch.zeros(n, dtype=torch.int8, device=device)
            self.gq_scales = torch.zeros(w["n_d"] * nbs, device=device)
            if w["stage"] == 3:
                # codes and scales beside each of the two gathered buffers
                self.gq_codes_l = [self.gq_codes, torch.zeros(n, dtype=torch.int8, device=device)]
                self.gq_scales_l = [self.gq_scales, torch.zeros(w["n_d"] * nbs, device=device)]
        if w.get("qgz"):
            # the int8 wire format of every gradient set (sender pass, untimed here)
            nbs = -(-self.plan.shard // 2048)
            # --row-pad applies to the int8 rows too (rounded to keep them 16-byte aligned)
            row16 = (w["psi"] + 15) // 16 * 16 + (w.get("row_pad", 0) + 15) // 16 * 16
            self.codes = [torch.empty(w["n_d"], row16, dtype=torch.int8, device=device) for _ in self.grads]
            n_dp = (w["n_d"] + 3) // 4 * 4
            self.qscales = [torch.empty(w["n_d"] * nbs * n_dp, device=device) for _ in self.grads]
            for k in range(len(self.grads)):
                self.quantize(k)
        if w.get("accum"):
            self.acc = torch.zeros(n, device=device)
        self.ws = torch.zeros(max(self.plan.workspace_bytes(self.hp), 256), dtype=torch.uint8, device=device)
        self.scalars = torch.zeros(256, dtype=torch.uint8, device=device)
        z.zero_scalars_init(self.scalars, scale)
        self.k = 0

    def quantize(self, k):
        """Sender side of the quantized gradient exchange for gradient set k."""
        self.z.zero_quantize_grads(self.plan.handle, [self.grads[k][r] for r in range(self.w["n_d"])], 2048,
                                   [self.codes[k][r] for r in range(self.w["n_d"])], self.qscales[k])

    def ranks(self, l):
        """Gradient set l's rank rows as the pointer array the library reads
        (built once: the sets never move)."""
        if not hasattr(self, "_rank_ptrs"):
            n_d = self.w["n_d"]
            self._rank_ptrs = [self.z.rank_ptrs([g[r] for r in range(n_d)]) for g in self.grads]
        return self._rank_ptrs[l % len(self.grads)]

    def code_ptrs(self, k):
        if not hasattr(self, "_code_ptrs"):
            n_d = self.w["n_d"]
            self._code_ptrs = [self.z.rank_ptrs([c[r] for r in range(n_d)]) for c in self.codes]
        return self._code_ptrs[k]

    def step(self):
        """One pass of the hot path through the public C ABI."""
        z, w = self.z, self.w
        h = self.plan.handle
        if w.get("accum"):
            self.step_accum()
            return
        if w["stage"] == 3:
            # one call for the stack: per layer its gather(s), then its fused
            # step (reduce-scatter of its ranks' gradients, Adam, 16-bit shards)
            z.zero_step_layers(self.hp, self.stack, w.get("gathers", 1), self.gathered, self.scalars,
                               gather_stream=self.gather_stream, gathered_codes=self.gq_codes_l,
                               gathered_scales=self.gq_scales_l)
            self.k += 1
            return
        for l in range(w["layers"]):
            gsel = self.k
            if w.get("qgz") and w.get("qgather"):
                k = gsel % len(self.grads)
                z.zero_step_fused_qgz_qgather(h, self.hp, self.code_ptrs(k), self.qscales[k], 2048, self.master[l],
                                              self.m[l], self.v[l], self.master[l], self.m[l], self.v[l],
                                              self.gq_codes, self.gq_scales, self.lp[l], self.scalars, self.ws)
            elif w.get("qgz"):
                k = gsel % len(self.grads)
                z.zero_step_fused_qgz(h, self.hp, self.code_ptrs(k), self.qscales[k], 2048,
                                      self.master[l], self.m[l], self.v[l], self.master[l], self.m[l], self.v[l],
                                      self.lp[l], self.scalars, self.ws)
            elif w.get("qgather"):
                z.zero_step_fused_qgather(h, self.hp, self.ranks(gsel), self.master[l], self.m[l], self.v[l],
                                          self.master[l], self.m[l], self.v[l], 2048, self.gq_codes, self.gq_scales,
                                          self.lp[l], self.scalars, self.ws)
            elif self.pingpong:
                z.zero_step_fused(h, self.hp, self.ranks(gsel), self.master[l], self.m[l], self.v[l],
                                  self.master2[l], self.m2[l], self.v2[l], self.lp[l], self.scalars, self.ws)
                self.master[l], self.master2[l] = self.master2[l], self.master[l]
                self.m[l], self.m2[l] = self.m2[l], self.m[l]
                self.v[l], self.v2[l] = self.v2[l], self.v[l]
            else:
                step = z.zero_step_fused_offload if self.offload else z.zero_step_fused
                step(h, self.hp, self.ranks(gsel), self.master[l], self.m[l], self.v[l], self.master[l], self.m[l],
                     self.v[l], self.lp[l], self.scalars, self.ws)
        self.k += 1

    def step_accum(self, sets=None):
        """One optimizer step over k micro-batches: k - 1 accumulations into
        the fp32 accumulator, then the step at the k-th."""
        z, w = self.z, self.w
        h = self.plan.handle
        k = w["accum"]
        for mu in range(k):
            g = self.ranks(self.k * k + mu if sets is None else sets)
            if mu < k - 1:
                z.zero_accumulate_grads(h, g, None if mu == 0 else self.acc, self.acc, self.scalars)
            else:
                z.zero_step_fused_accum(h, self.hp, g, self.acc, k, self.master[0], self.m[0], self.v[0],
                                        self.master[0], self.m[0], self.v[0], self.lp[0], self.scalars, self.ws)
        self.k += 1

    def parts_step(self, ev):
        """The clipped step through its parts, with an event between kernels:
        reduce-scatter (+ squared-norm partials) | finalize | Adam (+ epilogue)."""
        z = self.z
        h = self.plan.handle
        g = self.ghat
        ev[0].record()
        z.zero_reduce_scatter(h, self.ranks(self.k), self.hp, self.scalars, g, self.ws)
        ev[1].record()
        z.zero_grad_sqnorm(h, None, self.hp, self.scalars, self.ws)
        ev[2].record()
        z.zero_adam_shard_step(h, self.hp, g, self.master[0], self.m[0], self.v[0], self.lp[0], self.scalars)
        ev[3].record()
        self.k += 1


def l2_flush(torch, device, buf=[]):
    """Read 4x the L2 size: evicts the step's inputs with clean lines (a
    write would leave dirty lines whose write-back the step would pay for),
    and takes long enough that the host has enqueued the step before its
    start event."""
    if not buf:
        buf.append(torch.ones(4 * L2_BYTES // 4, dtype=torch.float32, device=device))
    buf[0].sum()


def gpu_arm(args, rank, world, device):
    import torch
    import zero_optimizer_step_02_gb300 as z
    w = workload_from_args(args)
    torch.cuda.set_device(device)
    job = Job(w, device)
    torch.cuda.synchronize()
    small = w["psi_total"] * w["bytes_per_param"] < 4 * L2_BYTES   # flush L2 between timed steps
    for _ in range(args.warmup):
        job.step()
    torch.cuda.synchronize()
    dist_barrier(world)

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    n0 = z.zero_launch_count()
    clocks.mark(0)
    if small:
        total_ms = 0.0
        for _ in range(args.steps):
            l2_flush(torch, device)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            job.step()
            b.record()
            torch.cuda.synchronize()
            total_ms += a.elapsed_time(b)
        launches = z.zero_launch_count() - n0
    else:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(args.steps):
            job.step()
        b.record()
        torch.cuda.synchronize()
        total_ms = a.elapsed_time(b)
        launches = z.zero_launch_count() - n0
    clocks.mark(1)
    clk = clocks.stop()
    warm_ms = graph_ms = None
    if small:
        # the same steps back to back with the inputs left in L2 (reported beside
        # the flushed number, which is the one `value` uses)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(args.steps):
            job.step()
        b.record()
        torch.cuda.synchronize()
        warm_ms = dist_max(a.elapsed_time(b), world) / args.steps
        # and replayed from a CUDA graph of 20 steps (no host launch cost per step)
        graph_ms = None
        if not w.get("accum") and not w.get("offload"):
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    for _ in range(20):
                        job.step()
            torch.cuda.current_stream().wait_stream(side)
            reps = max(1, args.steps // 20)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g.replay()
            torch.cuda.synchronize()
            a.record()
            for _ in range(reps):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            graph_ms = dist_max(a.elapsed_time(b), world) / (20 * reps)
    total_ms = dist_max(total_ms, world)
    ms_per_step = total_ms / args.steps
    value = world * w["psi_total"] * args.steps / (total_ms / 1e3)
    step_gbs = w["psi_total"] * w["bytes_per_param"] / (ms_per_step / 1e3) / 1e9

    # dominant kernel: per-kernel CUDA events on the launching stream
    peak, peak_kind = measured_hbm_peak()
    if w.get("accum"):
        # a middle micro-batch (accumulator read and written) and the step at
        # the last one, each timed alone back to back; the first repetition
        # is not counted
        n_rep = min(max(3, args.steps), 50)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_rep + 1)]
        torch.cuda.synchronize()
        for i, ev in enumerate(evs):
            ev[0].record()
            z.zero_accumulate_grads(job.plan.handle, job.ranks(i), job.acc, job.acc, job.scalars)
            ev[1].record()
            z.zero_step_fused_accum(job.plan.handle, job.hp, job.ranks(i + 1), job.acc, w["accum"], job.master[0],
                                    job.m[0], job.v[0], job.master[0], job.m[0], job.v[0], job.lp[0], job.scalars,
                                    job.ws)
            ev[2].record()
        torch.cuda.synchronize()
        t_acc = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evs[1:])
        t_fin = statistics.mean(ev[1].elapsed_time(ev[2]) for ev in evs[1:])
        kernel, kms, kbytes = "accumulate_grads", t_acc, (2 * w["n_d"] + 8) * w["psi"]
        breakdown = {"accumulate_grads": round(t_acc, 4), "step_accum": round(t_fin, 4)}
    elif w["clip"] > 0 and w["n_d"] > 4 and not (w.get("offload") or w.get("qgz") or w.get("qgather")):
        job.ghat = torch.zeros(job.plan.padded, device=device)
        n_rep = min(max(3, args.steps), 50)
        dur = [0.0, 0.0, 0.0]
        # enqueue every repetition back to back (one sync at the end) so the
        # host's launch latency never sits inside an interval; the first
        # repetition, which starts from an idle GPU, is not counted
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_rep + 1)]
        torch.cuda.synchronize()
        for ev in evs:
            job.parts_step(ev)
        torch.cuda.synchronize()
        for ev in evs[1:]:
            for i in range(3):
                dur[i] += ev[i].elapsed_time(ev[i + 1]) / n_rep
        names = ["reduce_scatter", "finalize", "adam_shard"]
        per_param = [2 * w["n_d"] + 4, 0.0, 30.0]
        k = max(range(3), key=lambda i: dur[i])
        kernel, kms, kbytes = names[k], dur[k], per_param[k] * w["psi"]
        breakdown = {names[i]: round(dur[i], 4) for i in range(3)}
    else:
        kernel = "fused_step" + ("_qgz" if w.get("qgz") else "") + ("_qgather" if w.get("qgather") else "")
        if w["clip"] > 0:
            kernel = "clipped_" + kernel     # both passes of the clipped step
        kms = ms_per_step / w["layers"] if w["stage"] != 3 else None
        if w["stage"] == 3:
            # time the per-layer fused step alone
            evs = []
            torch.cuda.synchronize()
            for _ in range(min(max(3, args.steps), 50) + 1):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                z.zero_step_fused(job.plan.handle, job.hp, job.ranks(0), job.master[0], job.m[0], job.v[0],
                                  job.master[0], job.m[0], job.v[0], job.lp[0], job.scalars, job.ws)
                b.record()
                evs.append((a, b))
            torch.cuda.synchronize()
            kms = statistics.mean(a.elapsed_time(b) for a, b in evs[1:])
            kbytes = (2 * w["n_d"] + 26) * w["psi"]
        else:
            kbytes = w["bytes_per_param"] * w["psi"]
        breakdown = None
    achieved = kbytes / (kms / 1e3) / 1e9
    tr = TRAFFIC.get((kernel, w["name"]))
    traffic = tr["bytes"] if tr and tr["src"] == kernel_source_hash() else None
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": kernel,
                "kernel_ms": round(kms, 4), "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)"}

    e2e = None if args.no_e2e else e2e_measure(job, w, args, device, world)
    if e2e is not None:
        # the link the end-to-end number is bound by, measured on this machine in
        # this run: the step's host-to-device rate against a plain 1 GiB copy's
        ms_e2e = w["psi_total"] * world / e2e["value"] * 1e3
        e2e["h2d_gbs"] = round(e2e["h2d_bytes_per_step"] / (ms_e2e / 1e3) / 1e9, 1)
        link = host_link_gbs(torch, device)
        e2e["host_link_gbs"] = link
        e2e["h2d_frac_of_link"] = round(e2e["h2d_gbs"] / link["h2d"], 4)
    sender = None
    if w.get("qgz"):
        # the sender pass (every rank quantizes its bf16 gradient): 2 + 1 + 4/2048 bytes per param per rank
        evs = []
        torch.cuda.synchronize()
        for k in range(min(max(3, args.steps), 50) + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            job.quantize(k % len(job.grads))
            b.record()
            evs.append((a, b))
        torch.cuda.synchronize()
        sms = statistics.mean(a.elapsed_time(b) for a, b in evs[1:])
        sbytes = w["n_d"] * w["psi"] * (3 + 4.0 / 2048)
        sender = {"ms": round(sms, 4), "gbs": round(sbytes / (sms / 1e3) / 1e9, 1),
                  "frac": round(sbytes / (sms / 1e3) / 1e9 / peak, 4)}
    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "gb300",
           "config": config_of(w, world),
           "step_gbs": round(step_gbs, 1), "step_frac_of_peak": round(step_gbs / peak, 4),
           "step_frac_of_nominal": round(step_gbs / NOMINAL_HBM_GBS, 4),
           "roofline": roofline, "gpu_launches": int(launches), "e2e": e2e, "clocks": clk}
    if breakdown:
        out["kernel_ms"] = breakdown
    if warm_ms is not None:
        out["warm_l2_ms_per_step"] = round(warm_ms, 4)
    if graph_ms is not None:
        out["warm_l2_cuda_graph_ms_per_step"] = round(graph_ms, 4)
    if sender:
        out["qgz_sender"] = sender
    if w.get("offload"):
        # the state's 12 bytes read + 12 written per parameter cross the CPU-GPU
        # link: against that link's duplex rate measured in this run
        link = host_link_gbs(torch, device)
        gbs = 24.0 * w["psi_total"] / (ms_per_step / 1e3) / 1e9
        out["offload_link_gbs"] = round(gbs, 1)
        out["host_link_gbs"] = link
        out["offload_link_frac"] = round(gbs / link["duplex"], 4)
    return out


def host_link_gbs(torch, device, nbytes=1 << 30, reps=3):
    """The CPU-GPU link measured here: pinned-host-to-device, device-to-host,
    and both at once on two streams (GB/s, both directions counted)."""
    h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=device)
    d_out = torch.ones(nbytes, dtype=torch.uint8, device=device)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps

    def both():
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)

    timed(both)
    h2d = nbytes / timed(lambda: d_in.copy_(h_in, non_blocking=True)) / 1e9
    d2h = nbytes / timed(lambda: h_out.copy_(d_out, non_blocking=True)) / 1e9
    duplex = 2 * nbytes / timed(both) / 1e9
    return {"h2d": round(h2d, 1), "d2h": round(d2h, 1), "duplex": round(duplex, 1)}


def e2e_measure(job, w, args, device, world):
    """Gradients from pinned host memory in, gathered parameters out, per step.

    The host-to-device copy of the next gradient set runs on a copy stream
    while the current one is reduced (two device buffers used in turn); every
    copy, every launch and the device-to-host read of each step's parameters
    lie inside the timed region."""
    import torch
    if w["layers"] > 1:
        return e2e_layers(job, w, args, world)
    if len(job.grads) < 2:
        return None
    z = job.z
    h = job.plan.handle
    qgz = bool(w.get("qgz"))
    if qgz:
        # the quantized exchange's wire format crosses the link: every rank's
        # int8 codes and fp32 block scales (the sender ran where the gradients are)
        dev_sets = [(job.codes[i], job.qscales[i]) for i in range(2)]
    else:
        dev_sets = [(job.grads[i],) for i in range(2)]
    host_in = []
    for t in dev_sets[0]:
        ht = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        ht.copy_(t)
        host_in.append(ht)
    host_out = torch.empty(job.lp[0].numel(), dtype=job.lp[0].dtype, pin_memory=True)
    steps = max(1, min(args.steps, 10))
    k = w.get("accum", 1)
    n_sets = steps * k                       # gradient sets crossing the link
    comp = torch.cuda.current_stream()
    copy_s = torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    used = [torch.cuda.Event(), torch.cuda.Event()]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def issue_copy(i):
        with torch.cuda.stream(copy_s):
            if i >= 2:
                copy_s.wait_event(used[i % 2])   # the pass that read this buffer is done
            for dst, src in zip(dev_sets[i % 2], host_in):
                dst.copy_(src, non_blocking=True)
            copied[i % 2].record(copy_s)

    torch.cuda.synchronize()
    a.record(comp)
    copy_s.wait_event(a)
    issue_copy(0)
    for i in range(n_sets):
        if i + 1 < n_sets:
            issue_copy(i + 1)
        comp.wait_event(copied[i % 2])
        mu = i % k
        if qgz:
            job.k = i % 2
            job.step()
        elif k > 1 and mu < k - 1:
            z.zero_accumulate_grads(h, job.ranks(i % 2), None if mu == 0 else job.acc, job.acc, job.scalars)
        elif k > 1:
            z.zero_step_fused_accum(h, job.hp, job.ranks(i % 2), job.acc, k, job.master[0], job.m[0], job.v[0],
                                    job.master[0], job.m[0], job.v[0], job.lp[0], job.scalars, job.ws)
        else:
            job.k = i % 2
            job.step()
        used[i % 2].record(comp)
        if mu == k - 1:
            host_out.copy_(job.lp[0], non_blocking=True)
    b.record(comp)
    torch.cuda.synchronize()
    ms = dist_max(a.elapsed_time(b), world)
    return {"value": world * w["psi"] * steps / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": k * sum(t.numel() * t.element_size() for t in host_in),
            "d2h_bytes_per_step": host_out.numel() * host_out.element_size(), "steps": steps,
            "overlap": "next gradient copy on a second stream",
            "inputs": "int8 codes + fp32 block scales of every rank" if qgz else "16-bit gradients of every rank"}


def e2e_layers(job, w, args, world):
    """The ZeRO-3 layer loop end to end: every step, every layer's rank
    gradients are copied from pinned host memory (a copy stream, layer after
    layer) and every layer's updated 16-bit shards copied back (a third
    stream).  One call of the layer loop per step; layer l's step waits for
    its gradients (grads_ready), and the next step's copy into layer l's
    buffers waits for layer l's step and the read-back of its shards
    (stepped), so copies, gathers and steps overlap across layers.  The
    host holds two of the layers' gradient sets (layer l copies from set
    l mod 2): the bytes crossing the link each step are every layer's."""
    import torch
    z = job.z
    L = w["layers"]
    steps = max(1, min(args.steps, 5))
    host_in = []
    for i in range(min(2, L)):
        ht = torch.empty(job.grads[i].shape, dtype=job.grads[i].dtype, pin_memory=True)
        ht.copy_(job.grads[i])
        host_in.append(ht)
    host_out = [torch.empty(job.lp[l].numel(), dtype=job.lp[l].dtype, pin_memory=True) for l in range(L)]
    comp = torch.cuda.current_stream()
    copy_s, out_s = torch.cuda.Stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(L)]
    stepped = [torch.cuda.Event() for _ in range(L)]
    read_back = [torch.cuda.Event() for _ in range(L)]
    stack = z.LayerStack([(job.plan.handle, job.ranks(l), job.master[l], job.m[l], job.v[l], job.lp[l], ready[l],
                           stepped[l]) for l in range(L)])
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(comp)
    copy_s.wait_event(a)
    for step in range(steps):
        for l in range(L):
            if step > 0:
                copy_s.wait_event(read_back[l])     # layer l's previous step and read-back are done
            with torch.cuda.stream(copy_s):
                job.grads[l].copy_(host_in[l % len(host_in)], non_blocking=True)
            ready[l].record(copy_s)
        z.zero_step_layers(job.hp, stack, w.get("gathers", 1), job.gathered, job.scalars,
                           gather_stream=job.gather_stream, gathered_codes=job.gq_codes_l,
                           gathered_scales=job.gq_scales_l)
        for l in range(L):
            out_s.wait_event(stepped[l])
            with torch.cuda.stream(out_s):
                host_out[l].copy_(job.lp[l], non_blocking=True)
            read_back[l].record(out_s)
    comp.wait_stream(copy_s)
    comp.wait_stream(out_s)
    b.record(comp)
    torch.cuda.synchronize()
    ms = dist_max(a.elapsed_time(b), world)
    return {"value": world * w["psi_total"] * steps / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": sum(g.numel() * g.element_size() for g in job.grads[:L]),
            "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in host_out), "steps": steps,
            "overlap": "per-layer copies on two copy streams, ordered by the layer loop's events",
            "inputs": "16-bit gradients of every rank of every layer (host holds two layers' sets, layer l "
                      "copies set l mod 2)"}


# ------------------------------------------------------------- CPU oracle arm
def oracle_sample(w, budget_s, max_steps=None):
    """Time the CPU oracle (as it stands, one thread) on a bounded sample of the
    workload: the same n_d, dtype and hyper-parameters on fewer parameters."""
    import numpy as np
    import oracle
    n_d = w["n_d"]
    # ~4M parameters at N_d = 8; fewer when a step reads more rank gradients
    psi = min(w["psi"], 4_000_000 * 8 // max(8, n_d * w.get("accum", 1)))
    rng = np.random.default_rng(1)
    dt = oracle.FP16 if w["gdt"] == "fp16" else oracle.BF16
    pdt = oracle.FP16 if w["pdt"] == "fp16" else oracle.BF16
    scale = 1024.0 if w["ls"] else 1.0
    rows = [oracle.f32_to_lp((rng.standard_normal(psi) * w["sigma"] * scale).astype(np.float32), dt)
            for _ in range(n_d)]
    S = oracle.shard_size(psi, n_d, w["pad"])
    st = oracle.State(np.zeros(n_d * S, np.float32), np.zeros(n_d * S, np.float32),
                      np.zeros(n_d * S, np.float32), oracle.new_scalars(scale))
    hp = oracle.hparams(lr=w["lr"], beta2=w["b2"], weight_decay=w["wd"], max_norm=w["clip"],
                        loss_scaling=w["ls"])
    lp = np.zeros(n_d * S, np.uint16)
    gath = np.zeros(psi, np.uint16)
    steps, t0 = 0, time.perf_counter()
    while True:
        if w.get("accum"):
            acc = None
            for _ in range(w["accum"] - 1):
                acc = oracle.accumulate_grads(rows, dt, acc)
            oracle.zero_step_accum(rows, dt, acc, w["accum"], hp, st, w["pad"], min(w["stage"], 3), lp_shards=lp,
                                   gathered=gath)
        elif w.get("qgz"):
            codes, scales = oracle.quantize_ranks(rows, psi, S, 2048)
            if w.get("qgather"):
                oracle.zero_step_qgz(codes, scales, 2048, hp, st, w["pad"], 3, psi, lp_shards=lp)
                oracle.quant_gather(lp, n_d, psi, S, 2048)
            else:
                oracle.zero_step_qgz(codes, scales, 2048, hp, st, w["pad"], min(w["stage"], 3), psi, lp_shards=lp,
                                     gathered=gath)
        elif w["stage"] == 3:
            # the ZeRO-3 layer step: the gather(s) of the 16-bit shards (block
            # int8 with qwZ), then the step
            for _ in range(w.get("gathers", 1)):
                if w.get("qgather"):
                    oracle.quant_gather(lp, n_d, psi, S, 2048)
                else:
                    oracle.all_gather_u16([lp[r * S:(r + 1) * S] for r in range(n_d)], psi, S)
            oracle.zero_step(rows, dt, hp, st, w["pad"], 3, param_dtype=pdt, lp_shards=lp)
        elif w.get("qgather"):
            # the step with its 16-bit output sharded, then the block-int8 gather of the shards
            oracle.zero_step(rows, dt, hp, st, w["pad"], 3, lp_shards=lp, gathered=gath)
            oracle.quant_gather(lp, n_d, psi, S, 2048)
        else:
            oracle.zero_step(rows, dt, hp, st, w["pad"], w["stage"], param_dtype=pdt, lp_shards=lp, gathered=gath)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps and steps >= max_steps):
            break
    return psi, n_d, steps, el


def reference_arm(args, rank, world):
    w = workload_from_args(args)
    if rank != 0:
        return None
    for _ in range(args.warmup):
        oracle_sample(w, 0.0, max_steps=1)
    # exactly K steps of the sample (no time budget)
    psi, n_d, steps, el = oracle_sample(w, float("inf"), max_steps=args.steps)
    value = psi * steps / el
    sample = "%d of %d params, n_d=%d, %d steps, single-threaded C oracle" % (psi, w["psi"], n_d, steps)
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * el / steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "impl": "reference", "config": config_of(w, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# -------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    return rank, world, local


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(x, world):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def build_parser():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200,
                    help="timed steps (the default makes the timed region long enough for several clock samples)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", type=int, default=4,
                    help="workload: 1 small ZeRO-2, 2 GPT-2-small clipped, 3 GPT-2 1.5B fp16, "
                         "4 ZeRO-3 8 Llama-3-8B layers (default: the largest), 5 the N_d sweep at 2^28")
    ap.add_argument("--nd", type=int, default=None)
    ap.add_argument("--qgather", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--psi", type=int, default=None, help="smaller parameter count (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--qgz", action="store_true", help="quantized gradient exchange (config 5)")
    ap.add_argument("--gathers", type=int, default=1, choices=[1, 2], help="ZeRO-3 gathers per layer and step")
    ap.add_argument("--offload", action="store_true", help="optimizer state in page-locked host memory")
    ap.add_argument("--accum", type=int, default=1, help="micro-batches per optimizer step (gradient accumulation)")
    ap.add_argument("--serial", action="store_true",
                    help="ZeRO-3: every gather on the step's stream (default: a second stream, overlapping)")
    ap.add_argument("--param-dtype", choices=["bf16", "fp16"], default=None,
                    help="16-bit parameter dtype (default bf16)")
    ap.add_argument("--stage", type=int, choices=[1, 2], default=None,
                    help="ZeRO stage of the ZeRO-1/2 workloads (same math, label and plan stage)")
    ap.add_argument("--row-pad", type=int, default=0,
                    help="extra elements between rank rows (breaks power-of-two rank strides)")
    return ap


def main():
    args = build_parser().parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_setup()
    if args.impl == "reference":
        out = reference_arm(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    import torch
    device = torch.device("cuda", local)
    out = gpu_arm(args, rank, world, device)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            w = workload_from_args(args)
            psi, n_d, steps, el = oracle_sample(w, args.cpu_budget)
            out["cpu_baseline"] = {"value": psi * steps / el, "unit": UNIT, "cores": 1, "kind": "oracle",
                                   "sample": "%d of %d params, n_d=%d, %d steps in %.1f s, single-threaded C "
                                             "oracle" % (psi, w["psi"], n_d, steps, el)}
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
