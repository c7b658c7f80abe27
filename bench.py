"""Benchmark of the paged-KV GQA attention hot path on GB300.

Default line (rank 0 prints one JSON line): the Qwen3-8B decode step, 36
layers of 64 sequences x 4096 tokens (16 query / 8 KV heads, head_dim 128,
bf16), one 1 GiB pool per layer (36 GiB of KV, far larger than L2).  One step
= for each layer: kv_cache_write of the 64 new tokens, then paged_attn_decode.
The same line carries two sub-lines with the same keys, each timed on its own:

  "prefill"      the Qwen3-0.6B mixed chunked-prefill step (budget 2048): per
                 layer, the write of 2048 new tokens, prefill of 3 chunks of
                 512 (prefixes 0, 512, 1536) beside the decode of 512
                 sequences; value in tokens/s, roofline = the prefill call on
                 the tensor cores (TFLOP/s);
  "decode_0_6b"  the Qwen3-0.6B decode step (8 sequences, 512..1024 tokens,
                 28 layers, fp16); value in KV GB/s.

Per line:
  value      the line's metric over the step time: CUDA events around K
             replays of a CUDA graph of one step, repeated until the timed
             region holds at least --min-seconds of GPU time (and at least 5
             repeats); ms_per_step is the median repeat / K;
  e2e        the same metric through the library calls with host buffers:
             each step copies every layer's inputs (and the step's metadata)
             from pinned host memory, replays the step's calls, and copies
             every layer's outputs back to pinned host memory;
  roofline   the dominant kernel timed alone (the step's attention calls back
             to back): algorithmic bytes (or FLOPs) per launch over its
             duration, against the measured HBM copy bandwidth (or dense bf16
             tensor throughput);
  cpu_baseline  the fp64 oracle on the host cores, on a bounded sample;
  clocks     nvidia-smi samples taken during the line's timed regions.

``--workload 2|3|5``, ``--kv``, ``--window``, ``--append``, ``--block-copy``
and ``--fused-write`` print single diagnostic lines instead.
``--impl reference`` times the oracle itself (the only reference this method
has) on the default line's workload and prints the same line with
"impl": "reference".  Multi-GPU (``torchrun --nproc-per-node N``) runs N
independent replicas (sequences are independent; no collective on the data
path): weak scaling.
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode paged-attn KV GB/s (% of GB300 HBM peak); prefill-chunk TFLOP/s; tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="each timed region repeats its K steps until it holds at least this much GPU time "
                         "(and at least 5 repeats); the median repeat gives ms_per_step")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle time budget of the cpu_baseline leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pools", type=int, default=0,
                    help="distinct layer pools held on the device (0 = the workload's default)")
    ap.add_argument("--kv", choices=["16bit", "int8", "fp8"], default="16bit",
                    help="the workload's 16-bit pool, or an int8 / fp8 (E4M3) pool (codes + one fp32 scale per "
                         "token and KV head) holding the same tokens quantised (workload 3: the 8-bit write, "
                         "prefill and decode)")
    ap.add_argument("--append", action="store_true",
                    help="decode workloads: each layer's KV write fused into its decode call "
                         "(paged_attn_decode_append) instead of a separate kv_cache_write")
    ap.add_argument("--no-early-pages", action="store_true",
                    help="decode workloads without a window: do not pass PA_DECODE_EARLY_PAGES. By "
                         "default each decode call fetches its cached pages before the preceding KV write has "
                         "finished, which the step allows: that write touches only each sequence's last page")
    ap.add_argument("--fused-combine", action="store_true",
                    help="decode calls with PA_DECODE_ZEROED_WORKSPACE: one launch over all SMs that merges "
                         "split sequences itself, instead of the plain plan (one cluster per sequence and KV "
                         "head when they fit, else split + combine kernels)")
    ap.add_argument("--balanced-prefill", action="store_true",
                    help="workload 3: the prefill as one launch balanced over the SMs "
                         "(pa_paged_attn_prefill_chunk_ex) instead of one CTA per query tile "
                         "(pa_paged_attn_prefill_chunk_window)")
    ap.add_argument("--overlap", action="store_true",
                    help="workload 3: each layer's prefill on a second stream beside its decode (same work)")
    ap.add_argument("--persistent-mixed", action="store_true",
                    help="workload 3 (16-bit pools, no window): each layer as ONE persistent launch "
                         "(pa_mixed_step: the write, then the prefill beside the decode on SMs split by their work)")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window of W keys for the attention calls of workloads 2, 3 and 4 (0 = none); "
                         "the bytes or FLOPs counted are those of the visible keys")
    ap.add_argument("--block-copy", action="store_true",
                    help="diagnostic line for the copy-on-write block copy: 64 (src, dst) pairs over the 28 "
                         "layer pools of the Qwen3-0.6B geometry (512 blocks of 16 x 8 x 128 fp16 each)")
    ap.add_argument("--fused-write", action="store_true",
                    help="diagnostic line for q/k RMSNorm + rotary embedding fused into the KV write: the mixed "
                         "step's 2048 new tokens (Qwen3-0.6B: 16 query / 8 KV heads, bf16) in each of 28 layers")
    ap.add_argument("--workload", type=int, default=4, choices=[2, 3, 4, 5],
                    help="4 = the Qwen3-8B 36-layer decode step (default; with the mixed prefill step and the "
                         "Qwen3-0.6B decode step as sub-lines); 2, 3, 5 = the Qwen3-0.6B decode step, the mixed "
                         "prefill step and the prefix-shared long tail alone")
    ap.add_argument("--no-sublines", action="store_true",
                    help="default workload: print the Qwen3-8B decode line without its two sub-lines")
    args = ap.parse_args(argv)
    if args.window < 0 or (args.window and (args.workload == 5 or args.kv != "16bit")):
        ap.error("--window takes W >= 0, with workloads 2, 3 and 4 on the 16-bit pool")
    if args.append and (args.window or args.kv != "16bit" or args.workload == 3):
        ap.error("--append applies to the 16-bit decode workloads 2, 4 and 5 without a window")
    args.early_pages = not args.no_early_pages and not args.window
    args.fused = args.fused_combine
    args.sublines = (args.workload == 4 and not args.no_sublines and args.kv == "16bit" and not args.window
                     and not args.append and not args.block_copy and not args.fused_write)
    return args


# ---- distributed plumbing (replicas only) -------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def reduce_max(x: float, device=None) -> float:
    """Max of a host float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and getattr(device, "type", "cpu") == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---- clocks during the timed region ----------------------------------------------------

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons every 200 ms (one
    `nvidia-smi -lms 200` process streaming rows) while the region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu              # nvidia-smi id: the device's UUID ("GPU-...") or an index
        self.rows = []
        self._proc = None
        self._t = None

    @staticmethod
    def gpu_id(device) -> str:
        """The nvidia-smi id of a torch device: its UUID when torch reports it
        (device indices inside the process need not match nvidia-smi's)."""
        import torch
        try:
            u = str(torch.cuda.get_device_properties(device).uuid)
            if u:
                return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        return str(device.index if device.index is not None else 0)

    def _read(self):
        for line in self._proc.stdout:
            line = line.strip()
            if line:
                self.rows.append([x.strip() for x in line.split(",")])

    def __enter__(self):
        try:
            self._proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                           "--format=csv,noheader,nounits", "-lms", "200"],
                                          stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self._proc = None
        return self

    def __exit__(self, *exc):
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=10)
            except Exception:
                self._proc.kill()
            self._t.join(timeout=10)
        return False

    def summary(self):
        num = lambda x: x.replace(".", "", 1).isdigit()
        sm = [float(r[1]) for r in self.rows if len(r) > 2 and num(r[1])]
        mx = [float(r[2]) for r in self.rows if len(r) > 2 and num(r[2])]
        pw = [float(r[3]) for r in self.rows if len(r) > 3 and num(r[3])]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons), "samples": len(self.rows)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def committed_traffic(kernel_sources, summary_name: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source: the summary records the sha256 of the source
    files (one name, or a tuple whose contents are hashed in that order)."""
    path = os.path.join(ROOT, "profiles", summary_name)
    names = (kernel_sources,) if isinstance(kernel_sources, str) else tuple(kernel_sources)
    try:
        text = open(path).read()
        src = b"".join(open(os.path.join(ROOT, "paged_kv_gqa_cache_gb300", "csrc", n), "rb").read() for n in names)
    except OSError:
        return None
    want = hashlib.sha256(src).hexdigest()[:16]
    m_hash = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", text)
    m_bytes = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != want:
        return None
    return int(m_bytes.group(1))


# ---- the workload ----------------------------------------------------------------------------

WORKLOADS = {
    2: ("Qwen3-0.6B decode step, 28 layers: 8 seqs, ctx U[512,1024], Hq=16, Hkv=8, d=128, fp16, "
        "512-block pool per layer", 28, 28),
    4: ("Qwen3-8B decode step, 36 layers: 64 seqs x 4096 ctx, Hq=32, Hkv=8, d=128, bf16, 16384-block pool "
        "(1 GiB K+V) per layer", 36, 36),
    5: ("Prefix-shared long-tail decode, Qwen3-8B geometry: 32 seqs sharing 13 blocks + suffixes "
        "log-U[16,32768], bf16; 4 distinct pools cycled over 8 calls", 4, 8),
}


class DecodeStep:
    """A decode step on device-resident inputs: for each of `calls` layers,
    kv_cache_write of the new tokens then paged_attn_decode (layer pools are
    cycled when fewer distinct pools than calls are held)."""

    def __init__(self, device, workload: int = 2, pools: int = 0, window: int = 0, append: bool = False,
                 early_pages: bool = False, fused: bool = False):
        import torch
        import paged_kv_gqa_cache_gb300 as pa
        import workloads
        self.pa = pa
        self.workload = workload
        self.window = window
        self.append = append
        self.early_pages = early_pages
        self.fused = fused            # PA_DECODE_ZEROED_WORKSPACE: one launch over all SMs
        self.desc, default_pools, self.L = WORKLOADS[workload]
        pools = pools or default_pools
        maker = workloads.BY_INDEX[workload]
        self.case = maker(device=device, n_layers=pools, nan_fill=False)
        c = self.case
        self.out = [torch.empty_like(q) for q in c.q]
        self.ws = pa.alloc_decode_workspace(c.q[0].shape[0], c.hq, c.hkv, c.max_context_len, device)
        lens = c.meta["decode_lens"]
        self.S = len(lens)
        self.dtype = c.dtype
        if c.meta.get("shared_prefix_blocks"):
            shared_tokens = 16 * c.meta["shared_prefix_blocks"]
            unique = sum(lens) - shared_tokens * (len(lens) - 1)
            self.decode_bytes_layer = workloads.decode_kv_bytes(lens, c.hkv, unique_tokens=unique)
        else:   # the visible rows: the last `window` of each sequence under a window
            self.decode_bytes_layer = workloads.decode_kv_bytes([min(n, window) if window else n for n in lens],
                                                                c.hkv)
        self.write_bytes_layer = 2 * c.k_new[0].numel() * 2 * 2     # K and V rows, read + write
        self.step_bytes = self.L * (self.decode_bytes_layer + self.write_bytes_layer)
        self.decode_kernels = 1 if fused else pa.decode_kernel_launches(self.S, c.hkv, c.max_context_len, window)
        # write, then the decode's kernels (the write runs inside the decode with append)
        self.kernels_per_step = self.L * ((0 if append else 1) + self.decode_kernels)

    # Layer l uses pool l % n_layers; its q, new K/V, output and the step's
    # metadata (slots, block tables, lengths) default to the resident tensors,
    # and the end-to-end run passes the ones it copied from the host.
    def write(self, l, kn=None, vn=None, meta=None):
        c, i = self.case, l % self.case.n_layers
        kn, vn = (c.k_new[i], c.v_new[i]) if kn is None else (kn, vn)
        slots = c.slot_mapping if meta is None else meta[0]
        self.pa.kv_cache_write(kn, vn, slots, c.k_cache[i], c.v_cache[i])

    def decode(self, l, q=None, out=None, kn=None, vn=None, meta=None):
        c, i = self.case, l % self.case.n_layers
        q = c.q[i] if q is None else q
        out = self.out[i] if out is None else out
        bt, ctx = (c.block_tables, c.context_lens) if meta is None else meta[1:]
        if self.append:
            kn, vn = (c.k_new[i], c.v_new[i]) if kn is None else (kn, vn)
            self.pa.paged_attn_decode_append(q, kn, vn, c.k_cache[i], c.v_cache[i], bt, ctx, c.scale, out=out,
                                             workspace=self.ws, max_context_len=c.max_context_len,
                                             early_pages=self.early_pages, zeroed_workspace=self.fused)
        elif self.window:
            self.pa.paged_attn_decode_window(q, c.k_cache[i], c.v_cache[i], bt, ctx, c.scale, self.window, out=out,
                                             workspace=self.ws, max_context_len=c.max_context_len,
                                             zeroed_workspace=self.fused)
        else:
            self.pa.paged_attn_decode(q, c.k_cache[i], c.v_cache[i], bt, ctx, c.scale, out=out, workspace=self.ws,
                                      max_context_len=c.max_context_len, early_pages=self.early_pages,
                                      zeroed_workspace=self.fused)

    def run(self):
        for l in range(self.L):
            if not self.append:
                self.write(l)
            self.decode(l)

    def run_decode_only(self):
        for l in range(self.L):
            self.decode(l)


class DecodeStepQ8(DecodeStep):
    """The same decode step over int8 pools ("Модуль 04: KV-кэш и арифметика
    памяти", section 5), or fp8 E4M3 pools (sections 5.1 and 5.4) with fp8:
    every cached token of each 16-bit layer pool is quantised once into an
    8-bit pool by the library's own write; each layer of the step then
    quantises the new tokens into their slots and decodes."""

    def __init__(self, device, workload: int = 2, pools: int = 0, fp8: bool = False, early_pages: bool = False,
                 fused: bool = False):
        import numpy as np
        import torch
        super().__init__(device, workload, pools, early_pages=early_pages, fused=fused)
        self.fp8 = fp8
        alloc = self.pa.alloc_pool_f8 if fp8 else self.pa.alloc_pool_q8
        self._write = self.pa.kv_cache_write_f8 if fp8 else self.pa.kv_cache_write_q8
        self._decode = self.pa.paged_attn_decode_f8 if fp8 else self.pa.paged_attn_decode_q8
        c = self.case
        bt = c.block_tables.cpu().numpy()
        slots = []
        for s_, n in enumerate(c.context_lens.cpu().numpy()):
            j = np.arange(int(n) - 1)                      # cached positions; the new token is written per step
            slots.append(bt[s_, j // 16].astype(np.int64) * 16 + j % 16)
        sl = torch.from_numpy(np.unique(np.concatenate(slots))).to(device)
        self.q8 = []
        for i in range(c.n_layers):
            pool = alloc(c.num_blocks, c.hkv, device)
            rows_k = c.k_cache[i].view(-1, c.hkv, 128)[sl].contiguous()
            rows_v = c.v_cache[i].view(-1, c.hkv, 128)[sl].contiguous()
            self._write(rows_k, rows_v, sl, *pool)
            self.q8.append(pool)
            del rows_k, rows_v
        torch.cuda.synchronize()
        per_token = c.hkv * (2 * 128 + 2 * 4)              # codes of K and V, one fp32 scale each
        self.decode_bytes_layer = self.decode_bytes_layer // (2 * c.hkv * 128 * 2) * per_token
        T = c.k_new[0].shape[0]
        self.write_bytes_layer = T * c.hkv * (2 * 128 * 2 + per_token // c.hkv)   # 16-bit rows in, codes out
        self.step_bytes = self.L * (self.decode_bytes_layer + self.write_bytes_layer)
        self.pool_bytes = sum(t.numel() * t.element_size() for t in self.q8[0])

    def write(self, l, kn=None, vn=None, meta=None):
        c, i = self.case, l % self.case.n_layers
        kn, vn = (c.k_new[i], c.v_new[i]) if kn is None else (kn, vn)
        self._write(kn, vn, c.slot_mapping if meta is None else meta[0], *self.q8[i])

    def decode(self, l, q=None, out=None, kn=None, vn=None, meta=None):
        c, i = self.case, l % self.case.n_layers
        bt, ctx = (c.block_tables, c.context_lens) if meta is None else meta[1:]
        self._decode(c.q[i] if q is None else q, *self.q8[i], bt, ctx, c.scale,
                     out=self.out[i] if out is None else out, workspace=self.ws, max_context_len=c.max_context_len,
                     early_pages=self.early_pages, zeroed_workspace=self.fused)


class MixedStep:
    """The Qwen3-0.6B mixed chunked-prefill step (budget 2048): per layer,
    kv_cache_write of 2048 new tokens, prefill of 3 chunks of 512 (prefixes 0,
    512, 1536) and decode of 512 sequences; 2 distinct pools cycled over 28."""

    def __init__(self, device, window: int = 0, overlap: bool = False, fused: bool = False, balanced: bool = False,
                 persistent: bool = False):
        import torch
        import paged_kv_gqa_cache_gb300 as pa
        import workloads
        self.pa, self.L, self.window, self.overlap, self.fused = pa, 28, window, overlap, fused
        # persistent: each layer is ONE launch (pa_mixed_step): the write, then the prefill beside the decode
        self.persistent = persistent and not window
        # overlap: each layer's prefill (tensor-bound) runs on a second stream beside its decode (HBM-bound)
        self.side = torch.cuda.Stream(device=device) if overlap else None
        self.case = c = workloads.qwen3_0_6b_mixed_step(device=device, n_layers=2, nan_fill=False)
        self.dtype = c.dtype
        self.out_d = [torch.empty_like(q) for q in c.q]
        self.out_p = [torch.empty_like(q) for q in c.q_chunks]
        self.ws = pa.alloc_decode_workspace(c.q[0].shape[0], c.hq, c.hkv, c.max_context_len, device)
        # the balanced prefill's workspace (zero-filled; every call leaves it zeroed)
        self.pws = pa.alloc_prefill_workspace(c.chunk_starts.numel(), c.hq, c.hkv, 512, device) if balanced else None
        self.flops_layer = workloads.prefill_flops(c.meta["chunks"], c.hq, window=window)
        self.tokens = c.slot_mapping.numel()
        lens = c.meta["decode_lens"]
        self.decode_bytes_layer = workloads.decode_kv_bytes([min(n, window) if window else n for n in lens], c.hkv)
        self.kernels_per_layer = 2 + (1 if fused else pa.decode_kernel_launches(len(lens), c.hkv, c.max_context_len,
                                                                                window))
        if self.persistent:  # the new tokens: the chunks' first, then one per decoding sequence
            self.mws = pa.alloc_mixed_step_workspace(len(lens), c.hq, c.hkv, device)
            self.chunk_tokens = sum(n for _, n in c.meta["chunks"])
            self.kernels_per_layer = 1

    def prefill(self, l, qp=None, out=None, meta=None):
        c, i = self.case, l % 2
        cs, cl, cbt, cctx = ((c.chunk_starts, c.chunk_lens, c.chunk_block_tables, c.chunk_context_lens)
                             if meta is None else meta[3:])
        self.pa.paged_attn_prefill_chunk_window(c.q_chunks[i] if qp is None else qp, cs, cl, c.k_cache[i],
                                                c.v_cache[i], cbt, cctx, c.scale, self.window,
                                                out=self.out_p[i] if out is None else out, max_chunk_len=512,
                                                workspace=self.pws)

    def layer(self, l, q=None, qp=None, kn=None, vn=None, out_d=None, out_p=None, meta=None):
        """One layer's calls; the end-to-end run passes the copies it made of
        the inputs and the metadata, and its own outputs."""
        import torch
        c, i = self.case, l % 2
        main = torch.cuda.current_stream()
        slots, bt, ctx = (c.slot_mapping, c.block_tables, c.context_lens) if meta is None else meta[:3]
        if self.persistent:
            cs, cl, cbt, cctx = ((c.chunk_starts, c.chunk_lens, c.chunk_block_tables, c.chunk_context_lens)
                                 if meta is None else meta[3:])
            kn, vn, tc = c.k_new[i] if kn is None else kn, c.v_new[i] if vn is None else vn, self.chunk_tokens
            self.pa.mixed_step(c.k_cache[i], c.v_cache[i], c.scale, self.mws, k_chunks=kn[:tc], v_chunks=vn[:tc],
                               chunk_slots=slots[:tc], q_chunks=c.q_chunks[i] if qp is None else qp, chunk_starts=cs,
                               chunk_lens=cl, chunk_block_tables=cbt, chunk_context_lens=cctx,
                               q=c.q[i] if q is None else q, k_dec=kn[tc:], v_dec=vn[tc:], block_tables=bt,
                               context_lens=ctx, out_chunks=self.out_p[i] if out_p is None else out_p,
                               out=self.out_d[i] if out_d is None else out_d, max_chunk_len=512)
            return
        self.pa.kv_cache_write(c.k_new[i] if kn is None else kn, c.v_new[i] if vn is None else vn, slots,
                               c.k_cache[i], c.v_cache[i])
        if self.side is not None:  # fork after the write, join before the next layer's write
            self.side.wait_stream(main)
            with torch.cuda.stream(self.side):
                self.prefill(l, qp, out_p, meta)
        else:
            self.prefill(l, qp, out_p, meta)
        self.pa.paged_attn_decode_window(c.q[i] if q is None else q, c.k_cache[i], c.v_cache[i], bt, ctx, c.scale,
                                         self.window, out=self.out_d[i] if out_d is None else out_d,
                                         workspace=self.ws, max_context_len=c.max_context_len,
                                         zeroed_workspace=self.fused)
        if self.side is not None:
            main.wait_stream(self.side)

    def run(self):
        for l in range(self.L):
            self.layer(l)

    def run_prefill_only(self):
        for l in range(self.L):
            self.prefill(l)


class MixedStepQ8(MixedStep):
    """The mixed step over int8 pools, or fp8 E4M3 pools with fp8 ("Модуль 04:
    KV-кэш и арифметика памяти", sections 5 and 5.4): every position of the
    two 16-bit layer pools quantised once by the library's own write; per layer
    the 8-bit write of the 2048 new tokens, the 8-bit prefill of the 3 chunks
    (pa_paged_attn_prefill_chunk_q8) and the 8-bit decode of the 512 sequences."""

    def __init__(self, device, fp8: bool = False, overlap: bool = False):
        import numpy as np
        import torch
        super().__init__(device, 0, overlap)
        self.fp8 = fp8
        pa, c = self.pa, self.case
        self._write8 = pa.kv_cache_write_f8 if fp8 else pa.kv_cache_write_q8
        self._prefill8 = pa.paged_attn_prefill_chunk_f8 if fp8 else pa.paged_attn_prefill_chunk_q8
        self._decode8 = pa.paged_attn_decode_f8 if fp8 else pa.paged_attn_decode_q8
        slots = []
        for bt, ctx in ((c.block_tables, c.context_lens), (c.chunk_block_tables, c.chunk_context_lens)):
            b = bt.cpu().numpy()
            for s_, n in enumerate(ctx.cpu().numpy()):
                j = np.arange(int(n))
                slots.append(b[s_, j // 16].astype(np.int64) * 16 + j % 16)
        sl = torch.from_numpy(np.unique(np.concatenate(slots))).to(device)
        alloc = pa.alloc_pool_f8 if fp8 else pa.alloc_pool_q8
        self.q8 = []
        for i in range(2):
            pool = alloc(c.num_blocks, c.hkv, device)
            self._write8(c.k_cache[i].view(-1, c.hkv, 128)[sl].contiguous(),
                         c.v_cache[i].view(-1, c.hkv, 128)[sl].contiguous(), sl, *pool)
            self.q8.append(pool)
        torch.cuda.synchronize()
        self.decode_bytes_layer = self.decode_bytes_layer // (2 * c.hkv * 128 * 2) * (c.hkv * (2 * 128 + 2 * 4))
        self.pool_bytes = sum(t.numel() * t.element_size() for t in self.q8[0])

    def prefill(self, l, qp=None, out=None, meta=None):
        c, i = self.case, l % 2
        cs, cl, cbt, cctx = ((c.chunk_starts, c.chunk_lens, c.chunk_block_tables, c.chunk_context_lens)
                             if meta is None else meta[3:])
        self._prefill8(c.q_chunks[i] if qp is None else qp, cs, cl, *self.q8[i], cbt, cctx, c.scale,
                       out=self.out_p[i] if out is None else out, max_chunk_len=512)

    def layer(self, l, q=None, qp=None, kn=None, vn=None, out_d=None, out_p=None, meta=None):
        import torch
        c, i = self.case, l % 2
        main = torch.cuda.current_stream()
        slots, bt, ctx = (c.slot_mapping, c.block_tables, c.context_lens) if meta is None else meta[:3]
        self._write8(c.k_new[i] if kn is None else kn, c.v_new[i] if vn is None else vn, slots, *self.q8[i])
        if self.side is not None:
            self.side.wait_stream(main)
            with torch.cuda.stream(self.side):
                self.prefill(l, qp, out_p, meta)
        else:
            self.prefill(l, qp, out_p, meta)
        self._decode8(c.q[i] if q is None else q, *self.q8[i], bt, ctx, c.scale,
                      out=self.out_d[i] if out_d is None else out_d, workspace=self.ws,
                      max_context_len=c.max_context_len)
        if self.side is not None:
            main.wait_stream(self.side)


def graph_of(fn, reps: int, stream):
    import torch
    fn()                                  # warm once outside capture (kernel attributes, caches)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                fn()
    torch.cuda.synchronize()
    return g


def time_replays(g, n: int, stream) -> float:
    """Milliseconds for n replays of graph g, by CUDA events on its stream."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1)


def timed_repeats(one_repeat, min_seconds: float, min_reps: int = 5, max_reps: int = 5000):
    """Run one_repeat() (it returns the milliseconds of K timed steps) until the
    repeats hold at least min_seconds of GPU time and number at least min_reps.
    Returns the per-repeat milliseconds."""
    reps = [one_repeat()]
    while (len(reps) < min_reps or sum(reps) < 1e3 * min_seconds) and len(reps) < max_reps:
        reps.append(one_repeat())
    return reps


def timing_summary(reps, steps: int) -> dict:
    return {"repeats": len(reps), "steps_per_repeat": steps, "timed_region_s": round(sum(reps) / 1e3, 3),
            "ms_per_step_min": round(min(reps) / steps, 5), "ms_per_step_max": round(max(reps) / steps, 5)}


def _e2e_run(L, layer_inputs, meta, layer_outputs, calls, steps, warmup, stream, min_seconds):
    """The end-to-end leg shared by the lines: per step one copy of every
    layer's inputs and of the step's metadata from pinned host memory into one
    staging buffer, the step's library calls (captured once as a CUDA graph,
    reading the staged copies), and one copy of every layer's outputs into
    pinned host memory.  layer_inputs[l] and layer_outputs[l] are tuples of
    tensors; calls(l, inputs, meta, outputs) enqueues layer l's calls.
    Returns (median ms per step, h2d bytes, d2h bytes, repeats, host outputs)."""
    import torch
    dev = layer_outputs[0][0].device
    align = lambda x: (x + 255) // 256 * 256
    nbytes = lambda t: t.numel() * t.element_size()
    parts, off = [], 0
    for l in range(L):
        for src in layer_inputs[l]:
            parts.append((src, off))
            off = align(off + nbytes(src))
    for src in meta:
        parts.append((src, off))
        off = align(off + nbytes(src))
    host_in = torch.empty(off, dtype=torch.uint8).pin_memory()
    dev_in = torch.empty(off, dtype=torch.uint8, device=dev)
    views = []
    for src, o in parts:
        host_in[o:o + nbytes(src)].copy_(src.contiguous().view(torch.uint8).view(-1).cpu())
        views.append(dev_in[o:o + nbytes(src)].view(src.dtype).view(src.shape))
    out_parts, ooff = [], 0
    for l in range(L):
        for like in layer_outputs[l]:
            out_parts.append((like, ooff))
            ooff = align(ooff + nbytes(like))
    dev_out = torch.empty(ooff, dtype=torch.uint8, device=dev)
    host_out = torch.empty(ooff, dtype=torch.uint8).pin_memory()
    outs = [dev_out[o:o + nbytes(t)].view(t.dtype).view(t.shape) for t, o in out_parts]
    n_in, n_out = len(layer_inputs[0]), len(layer_outputs[0])
    meta_views = tuple(views[L * n_in:])

    def step_calls():
        for l in range(L):
            calls(l, views[n_in * l:n_in * (l + 1)], meta_views, outs[n_out * l:n_out * (l + 1)])

    dev_in.copy_(host_in)               # staged once before the graph's warm-up call and capture
    torch.cuda.synchronize()
    graph = graph_of(step_calls, 1, stream)

    def one():
        dev_in.copy_(host_in, non_blocking=True)
        graph.replay()
        host_out.copy_(dev_out, non_blocking=True)

    def one_repeat():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                one()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            one()
    torch.cuda.synchronize()
    reps = timed_repeats(one_repeat, min_seconds)
    host_views = [host_out[o:o + nbytes(t)].view(t.dtype).view(t.shape) for t, o in out_parts]
    host_layers = [tuple(host_views[n_out * l:n_out * (l + 1)]) for l in range(L)]
    return statistics.median(reps) / steps, off, ooff, len(reps), host_layers


def e2e_measure(step: DecodeStep, steps: int, warmup: int, stream, min_seconds: float = 0.0):
    """Same metric through the public API with host buffers, the way a serving
    loop runs a decode step: per step one host-to-device copy, from pinned host
    memory, of every layer's q and new K/V rows and of the step's slots, block
    tables and lengths; the step's library calls (write + decode per layer,
    replayed as a CUDA graph of those calls); one device-to-host copy of every
    layer's output into pinned host memory.  Every layer has its own inputs
    and output; the pools are the resident ones the step cycles."""
    c, L, n = step.case, step.L, step.case.n_layers
    append = getattr(step, "append", False)

    def calls(l, ins, meta, outs):
        q, kn, vn = ins
        if not append:
            step.write(l, kn, vn, meta=meta)
        step.decode(l, q=q, out=outs[0], kn=kn, vn=vn, meta=meta)

    ms, h2d, d2h, reps, host = _e2e_run(
        L, [(c.q[l % n], c.k_new[l % n], c.v_new[l % n]) for l in range(L)],
        (c.slot_mapping, c.block_tables, c.context_lens), [(step.out[l % n],) for l in range(L)], calls, steps,
        warmup, stream, min_seconds)
    step.e2e_outputs = [h[0] for h in host]      # the outputs of the last step as they reached the host
    return ms, h2d, d2h


def e2e_measure_mixed(step: MixedStep, steps: int, warmup: int, stream, min_seconds: float = 0.0):
    """The end-to-end leg of the mixed step: per step every layer's decode
    queries, chunk queries and new K/V rows plus the step's metadata (slots,
    decode tables and lengths, chunk starts, lengths, tables and context
    lengths) from pinned host memory, the step's calls, and every layer's
    decode and prefill outputs back to pinned host memory."""
    c, L = step.case, step.L

    def calls(l, ins, meta, outs):
        q, qp, kn, vn = ins
        step.layer(l, q=q, qp=qp, kn=kn, vn=vn, out_d=outs[0], out_p=outs[1], meta=meta)

    ms, h2d, d2h, reps, host = _e2e_run(
        L, [(c.q[l % 2], c.q_chunks[l % 2], c.k_new[l % 2], c.v_new[l % 2]) for l in range(L)],
        (c.slot_mapping, c.block_tables, c.context_lens, c.chunk_starts, c.chunk_lens, c.chunk_block_tables,
         c.chunk_context_lens), [(step.out_d[l % 2], step.out_p[l % 2]) for l in range(L)], calls, steps, warmup,
        stream, min_seconds)
    step.e2e_outputs = host
    return ms, h2d, d2h


def _u16(t):
    import numpy as np
    import torch
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def cpu_baseline(step: DecodeStep, seconds: float):
    """The fp64 oracle, as it stands, on the host cores: the workload's decode
    layer calls in order, repeated until about `seconds` of wall time (a
    bounded sample of the same work, scaled to GB/s).  At most two distinct
    layer pools are copied to the host (each layer's pool is as large as
    every other's; a 1 GiB pool per layer would not fit 36 times)."""
    import oracle
    c = step.case
    threads = os.cpu_count() or 1
    bt, ctx = c.block_tables.cpu().numpy(), c.context_lens.cpu().numpy()
    odt = oracle.BF16 if c.dtype == "bf16" else oracle.F16
    q8 = getattr(step, "q8", None)
    window = getattr(step, "window", 0)
    pools = min(c.n_layers, 2)
    inputs = {}

    def host(i):   # a layer's host copies, made once on first use, outside the timed calls
        if i not in inputs:
            if q8 is not None:
                inputs[i] = (_u16(c.q[i]), [t.cpu().numpy() for t in q8[i]])
            else:
                inputs[i] = (_u16(c.q[i]), _u16(c.k_cache[i]), _u16(c.v_cache[i]))
        return inputs[i]

    done_bytes, t_total, calls = 0, 0.0, 0
    while t_total < seconds:
        for l in range(step.L):
            x = host(l % pools)
            t0 = time.perf_counter()
            if q8 is not None:
                (oracle.paged_attn_decode_f8 if step.fp8 else oracle.paged_attn_decode_q8)(
                    x[0], *x[1], bt, ctx, c.scale, odt, num_threads=threads)
            elif window:
                oracle.paged_attn_decode_window(x[0], x[1], x[2], bt, ctx, c.scale, window, odt, num_threads=threads)
            else:
                oracle.paged_attn_decode(x[0], x[1], x[2], bt, ctx, c.scale, odt, num_threads=threads)
            t_total += time.perf_counter() - t0
            done_bytes += step.decode_bytes_layer
            calls += 1
            if t_total >= seconds:
                break
    return {"value": round(done_bytes / t_total / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{calls} decode layer calls of the workload in step order over {pools} distinct layer "
                      f"pools (fp64 C oracle, {threads} threads), {t_total:.2f} s"}


def cpu_baseline_mixed(step: MixedStep, seconds: float):
    """The fp64 oracle on the host cores for the mixed step: per layer the KV
    write, the prefill of the three chunks and the decode of the 512
    sequences, layers in step order until about `seconds` of wall time; scaled
    to tokens/s of the 28-layer step (2048 tokens per step), with the prefill
    part also in TFLOP/s."""
    import numpy as np
    import oracle
    c = step.case
    threads = os.cpu_count() or 1
    bt, ctx = c.block_tables.cpu().numpy(), c.context_lens.cpu().numpy()
    cs, cl = c.chunk_starts.cpu().numpy(), c.chunk_lens.cpu().numpy()
    cbt, cctx = c.chunk_block_tables.cpu().numpy(), c.chunk_context_lens.cpu().numpy()
    slots = c.slot_mapping.cpu().numpy()
    q8 = getattr(step, "q8", None)
    odt = oracle.BF16 if c.dtype == "bf16" else oracle.F16
    if q8 is not None:
        hosts = [dict(p8=[t.cpu().numpy().copy() for t in q8[i]], kn=_u16(c.k_new[i]), vn=_u16(c.v_new[i]),
                      q=_u16(c.q[i]), qp=_u16(c.q_chunks[i])) for i in range(2)]
        w8 = oracle.kv_cache_write_f8 if step.fp8 else oracle.kv_cache_write_q8
        p8 = oracle.paged_attn_prefill_f8 if step.fp8 else oracle.paged_attn_prefill_q8
        d8 = oracle.paged_attn_decode_f8 if step.fp8 else oracle.paged_attn_decode_q8
    else:
        hosts = [dict(k=_u16(c.k_cache[i]).copy(), v=_u16(c.v_cache[i]).copy(), kn=_u16(c.k_new[i]),
                      vn=_u16(c.v_new[i]), q=_u16(c.q[i]), qp=_u16(c.q_chunks[i])) for i in range(2)]
    t_total, t_pre, layers = 0.0, 0.0, 0
    while t_total < seconds:
        x = hosts[layers % 2]
        if q8 is not None:
            t0 = time.perf_counter()
            w8(*x["p8"], x["kn"], x["vn"], odt, slots)
            t1 = time.perf_counter()
            p8(x["qp"], *x["p8"], cs, cl, cbt, cctx, c.scale, odt, num_threads=threads)
            t2 = time.perf_counter()
            d8(x["q"], *x["p8"], bt, ctx, c.scale, odt, num_threads=threads)
            t3 = time.perf_counter()
            t_total += t3 - t0
            t_pre += t2 - t1
            layers += 1
            continue
        t0 = time.perf_counter()
        oracle.kv_cache_write(x["k"], x["v"], x["kn"], x["vn"], slots)
        t1 = time.perf_counter()
        if step.window:
            oracle.paged_attn_prefill_window(x["qp"], x["k"], x["v"], cs, cl, cbt, cctx, c.scale, step.window,
                                             oracle.BF16, num_threads=threads)
        else:
            oracle.paged_attn_prefill(x["qp"], x["k"], x["v"], cs, cl, cbt, cctx, c.scale, oracle.BF16,
                                      num_threads=threads)
        t2 = time.perf_counter()
        if step.window:
            oracle.paged_attn_decode_window(x["q"], x["k"], x["v"], bt, ctx, c.scale, step.window, oracle.BF16,
                                            num_threads=threads)
        else:
            oracle.paged_attn_decode(x["q"], x["k"], x["v"], bt, ctx, c.scale, oracle.BF16, num_threads=threads)
        t3 = time.perf_counter()
        t_total += t3 - t0
        t_pre += t2 - t1
        layers += 1
    tokens_per_s = (layers / step.L) * step.tokens / t_total
    return {"value": round(tokens_per_s, 3), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "prefill_tflops": round(layers * step.flops_layer / t_pre / 1e12, 6),
            "sample": f"{layers} of the step's {step.L} layers (write of {step.tokens} tokens, prefill of the 3 "
                      f"chunks, decode of {len(ctx)} sequences"
                      + (f", over {'E4M3' if step.fp8 else 'int8'} pools" if q8 is not None else "")
                      + f"; fp64 C oracle, {threads} threads), "
                      f"{t_total:.2f} s, scaled to the {step.L}-layer step"}


def _device_error_check(pa):
    st, detail = pa.get_device_error()
    if st != 0:
        raise RuntimeError(f"device error {pa.STATUS.get(st, st)} at {detail}")


def decode_line(args, dev, pa, workload: int, kv: str = "16bit", window: int = 0, append: bool = False,
                early_pages: bool = True, pools: int = 0, cpu: bool = True) -> dict:
    """The JSON line of one decode workload (steps of write + decode per layer)."""
    import torch
    rank, world, _ = dist_env()
    step = (DecodeStepQ8(dev, workload, pools, kv == "fp8", early_pages, args.fused) if kv != "16bit"
            else DecodeStep(dev, workload, pools, window, append, early_pages, args.fused))
    stream = torch.cuda.Stream(device=dev)
    g_step = graph_of(step.run, 1, stream)
    g_dec = graph_of(step.run_decode_only, 1, stream)
    _device_error_check(pa)

    # warm-up, then repeats of K timed steps bracketed by barrier + synchronize
    time_replays(g_step, max(args.warmup, 3), stream)
    barrier(dev)
    torch.cuda.synchronize()
    with ClockSampler(ClockSampler.gpu_id(dev)) as clk:
        reps = timed_repeats(lambda: time_replays(g_step, args.steps, stream), args.min_seconds)
        torch.cuda.synchronize()
        barrier(dev)
        # the dominant kernel alone: the step's decode calls, back to back
        dec_reps = timed_repeats(lambda: time_replays(g_dec, args.steps, stream), args.min_seconds / 2)
        e2e_ms, h2d, d2h = e2e_measure(step, args.steps, max(args.warmup, 3), stream, args.min_seconds / 2)
    ms_step = reduce_max(statistics.median(reps) / args.steps, dev)
    e2e_ms = reduce_max(e2e_ms, dev)
    _device_error_check(pa)
    hbm, bf16, peak_kind = measured_peaks()
    value = world * step.step_bytes / (ms_step * 1e-3) / 1e9

    dec_launch_ms = statistics.median(dec_reps) / args.steps / step.L
    # with append the decode call also moves the new rows (read, written into the pool)
    launch_bytes = step.decode_bytes_layer + (step.write_bytes_layer if getattr(step, "append", False) else 0)
    achieved = launch_bytes / (dec_launch_ms * 1e-3) / 1e9

    q8 = isinstance(step, DecodeStepQ8)
    pool_mib = (step.pool_bytes if q8 else 2 * step.case.k_cache[0].numel() * 2) / 2**20
    win = getattr(step, "window", 0)
    tag = (("_f8" if step.fp8 else "_q8") if q8 else
           (f"_window{win}" if win else ("_append" if getattr(step, "append", False) else "")))
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "data": "synthetic",
        "dtype": ("fp8_e4m3" if step.fp8 else "int8") if q8 else step.dtype,
        "config": {"workload": step.desc + (f", {'fp8 E4M3' if step.fp8 else 'int8'} KV pool (codes + one fp32 "
                                            f"scale per token and KV head), {step.dtype} q and out" if q8 else "")
                               + (f", sliding window of {win} keys (bytes of the visible rows)" if win else "")
                               + (", KV write fused into the decode call" if getattr(step, "append", False) else "")
                               + (", cached pages fetched before the preceding write ends (PA_DECODE_EARLY_PAGES)"
                                  if getattr(step, "early_pages", False) else "")
                               + (", one decode launch over all SMs merging split sequences itself "
                                  "(PA_DECODE_ZEROED_WORKSPACE)" if step.fused else ""),
                   "global_batch": step.S * world, "seq_len": step.case.max_context_len,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 ({step.case.n_layers} distinct pools of {pool_mib:.0f} MiB "
                         f"cycled over {step.L} calls per step)",
                   "timing": "CUDA events around K replays of a CUDA graph of one step, repeated; median repeat"},
        "timing": timing_summary(reps, args.steps),
        "pct_of_hbm_peak": round(100.0 * value / world / hbm, 1),
        "tokens_per_s": round(world * step.S / (ms_step * 1e-3), 1),
        "gpu_launches": step.kernels_per_step * args.steps * len(reps),
        "e2e": {"value": round(world * step.step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 3), "peak_kind": peak_kind,
                     "kernel": "paged_attn_decode" + tag + " per layer ("
                               + ("one launch over all SMs, split sequences merged in it" if step.fused else
                                  "one cluster per sequence and KV head" if step.decode_kernels == 1
                                  else "split + combine") + ")",
                     "bytes_per_launch": launch_bytes, "launch_ms": round(dec_launch_ms, 5),
                     "launches_timed": step.L * args.steps * len(dec_reps),
                     "traffic": committed_traffic(("decode.cu", "decode_kernel.cuh"), f"decode{tag}_workload{workload}.md")},
        "clocks": clk.summary(),
    }
    if rank == 0 and cpu and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(step, args.cpu_seconds)
    del step, g_step, g_dec
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


def mixed_line(args, dev, pa, window: int = 0, overlap: bool = False, cpu: bool = True, kv: str = "16bit") -> dict:
    """The JSON line of the mixed chunked-prefill step (28 layers), over 16-bit
    pools or (kv "int8" / "fp8") 8-bit ones."""
    import torch
    rank, world, _ = dist_env()
    q8 = kv != "16bit"
    step = (MixedStepQ8(dev, kv == "fp8", overlap) if q8 else
            MixedStep(dev, window, overlap, args.fused, balanced=args.balanced_prefill,
                      persistent=args.persistent_mixed))
    stream = torch.cuda.Stream(device=dev)
    g_step = graph_of(step.run, 1, stream)
    g_pre = graph_of(step.run_prefill_only, 1, stream)
    _device_error_check(pa)
    time_replays(g_step, max(args.warmup, 3), stream)
    barrier(dev)
    torch.cuda.synchronize()
    with ClockSampler(ClockSampler.gpu_id(dev)) as clk:
        reps = timed_repeats(lambda: time_replays(g_step, args.steps, stream), args.min_seconds)
        torch.cuda.synchronize()
        barrier(dev)
        pre_reps = timed_repeats(lambda: time_replays(g_pre, args.steps, stream), args.min_seconds / 2)
        e2e_ms, h2d, d2h = e2e_measure_mixed(step, args.steps, max(args.warmup, 3), stream, args.min_seconds / 2)
    ms_step = reduce_max(statistics.median(reps) / args.steps, dev)
    e2e_ms = reduce_max(e2e_ms, dev)
    ms_pre = statistics.median(pre_reps) / args.steps / step.L
    _device_error_check(pa)
    hbm, bf16, peak_kind = measured_peaks()
    tflops = step.flops_layer / (ms_pre * 1e-3) / 1e12
    line = {
        "metric": "mixed chunked-prefill step tokens/s; prefill-chunk TFLOP/s",
        "value": round(world * step.tokens / (ms_step * 1e-3), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": (("fp8_e4m3" if step.fp8 else "int8") if q8 else "bf16"), "data": "synthetic",
        "config": {"workload": "Qwen3-0.6B mixed chunked-prefill step, 28 layers: chunks (0,512), (512,512), "
                               "(1536,512) + 512 decode seqs ctx U[16,1024], Hq=16, Hkv=8, d=128, bf16; "
                               "2 distinct pools cycled"
                               + ((f"; {'fp8 E4M3' if step.fp8 else 'int8'} KV pools (codes + one fp32 scale per "
                                   "token and KV head): 8-bit write, prefill and decode, bf16 q and out") if q8
                                  else "")
                               + (f"; sliding window of {window} keys (FLOPs of the visible pairs)" if window else "")
                               + ("; each layer's prefill on a second stream beside its decode"
                                  if overlap and not getattr(step, "persistent", False) else "")
                               + ("; each layer as one persistent launch (pa_mixed_step: the chunks' write, then "
                                  "their prefill, beside the decode that appends the sequences' new tokens)"
                                  if getattr(step, "persistent", False) else "")
                               + ("; prefill balanced over the SMs (pa_paged_attn_prefill_chunk_ex)"
                                  if step.pws is not None else "")
                               + ("; decode as one launch over all SMs (PA_DECODE_ZEROED_WORKSPACE)"
                                  if step.fused else ""),
                   "global_batch": 515 * world, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (2 pools of {:.0f} MiB cycled over 28 layers)".format(
                       (step.pool_bytes if q8 else 2 * step.case.k_cache[0].numel() * 2) / 2**20),
                   "timing": "CUDA events around K replays of a CUDA graph of one step, repeated; median repeat"},
        "timing": timing_summary(reps, args.steps),
        "decode_kv_gbs": round(step.L * step.decode_bytes_layer / (ms_step * 1e-3) / 1e9, 1),
        "gpu_launches": step.L * step.kernels_per_layer * args.steps * len(reps),
        "e2e": {"value": round(world * step.tokens / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
        "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": bf16, "unit": "TFLOP/s",
                     "frac": round(tflops / bf16, 3), "peak_kind": peak_kind,
                     "kernel": (f"paged_attn_prefill_chunk_q8 ({'E4M3' if step.fp8 else 'int8'} pool, tcgen05)"
                                if q8 else "paged_attn_prefill_chunk" + ("_ex (balanced)" if step.pws is not None
                                                                         else ""))
                               + (f" window W={window}" if window else "") + " per layer",
                     "flops_per_launch": step.flops_layer,
                     "launch_ms": round(ms_pre, 5), "launches_timed": step.L * args.steps * len(pre_reps),
                     "traffic": (committed_traffic(("prefill8.cu", "prefill_kernel.cuh"), f"prefill8_{kv}_workload3.md")
                                 if q8 else
                                 committed_traffic(("prefill.cu", "prefill_kernel.cuh"),
                                                   f"prefill{f'_window{window}' if window else ''}_workload3.md"))},
        "clocks": clk.summary(),
    }
    if rank == 0 and cpu and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_mixed(step, args.cpu_seconds)
    del step, g_step, g_pre
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init("nccl")
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_gqa_cache_gb300 as pa
    if args.block_copy:
        return run_block_copy(args, dev, pa)
    if args.fused_write:
        return run_fused_write(args, dev, pa)
    if args.workload == 3:
        line = mixed_line(args, dev, pa, args.window, args.overlap, kv=args.kv)
    else:
        line = decode_line(args, dev, pa, args.workload, args.kv, args.window, args.append, args.early_pages,
                           args.pools)
    if args.sublines:
        line["prefill"] = mixed_line(args, dev, pa, overlap=True)
        line["decode_0_6b"] = decode_line(args, dev, pa, 2, early_pages=args.early_pages)
        # the 8-bit pools: the 8B decode layer over int8 and E4M3 codes, the mixed step over int8 codes
        line["decode_8b_int8"] = decode_line(args, dev, pa, 4, kv="int8", early_pages=args.early_pages, pools=4)
        line["decode_8b_fp8"] = decode_line(args, dev, pa, 4, kv="fp8", early_pages=args.early_pages, pools=4)
        line["prefill_int8"] = mixed_line(args, dev, pa, kv="int8")
        line["gpu_launches_sublines"] = sum(line[k]["gpu_launches"] for k in
                                            ("prefill", "decode_0_6b", "decode_8b_int8", "decode_8b_fp8",
                                             "prefill_int8"))
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_block_copy(args, dev, pa):
    """Diagnostic line for the copy-on-write block copy over every layer."""
    import numpy as np
    import torch
    rank, world, _ = dist_env()
    layers, nb, hkv, npairs = 28, 512, 8, 64
    g = torch.Generator(device=dev).manual_seed(7)
    pools = [(torch.randn((nb, 16, hkv, 128), generator=g, device=dev).to(torch.float16),
              torch.randn((nb, 16, hkv, 128), generator=g, device=dev).to(torch.float16)) for _ in range(layers)]
    perm = np.random.default_rng(7).permutation(nb)
    # alternate two disjoint pair sets so consecutive copies never touch the same blocks
    sets = [torch.from_numpy(np.stack([perm[i * 2 * npairs:i * 2 * npairs + npairs],
                                       perm[i * 2 * npairs + npairs:(i + 1) * 2 * npairs]], 1).astype(np.int32)
                             ).to(dev) for i in range(2)]
    stream = torch.cuda.Stream(device=dev)
    launches = -(-layers // 64)

    def step():
        for pr in sets:
            pa.kv_block_copy(pools, pr)

    g_step = graph_of(step, 1, stream)
    _device_error_check(pa)
    time_replays(g_step, max(args.warmup, 3), stream)
    barrier(dev)
    torch.cuda.synchronize()
    with ClockSampler(ClockSampler.gpu_id(dev)) as clk:
        reps = timed_repeats(lambda: time_replays(g_step, args.steps, stream), args.min_seconds)
        ms_step = statistics.median(reps) / args.steps
    ms_step = reduce_max(ms_step, dev)
    _device_error_check(pa)
    hbm, _, peak_kind = measured_peaks()
    block_bytes = 16 * hkv * 128 * 2
    step_bytes = 2 * npairs * layers * 2 * block_bytes * 2     # 2 sets x pairs x layers x (K, V) x (read + write)
    gbs = step_bytes / (ms_step * 1e-3) / 1e9
    line = {
        "metric": "KV block copy GB/s (copy-on-write, every layer)", "value": round(world * gbs, 1),
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic",
        "config": {"workload": f"copy-on-write of {npairs} blocks x 2 pair sets over {layers} layer pools "
                               f"({nb} blocks of 16 x {hkv} x 128 fp16 each, 896 MiB in total)",
                   "l2": "each step touches 2 x 64 x 28 distinct 32 KB block copies (117 MB read, 117 MB "
                         "written); the pools (896 MiB) exceed L2",
                   "timing": "CUDA events around a CUDA graph of one step, replayed K times"},
        "gpu_launches": 2 * launches * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs / hbm, 3), "peak_kind": peak_kind, "kernel": "kv_block_copy",
                     "bytes_per_launch": step_bytes // 2, "launch_ms": round(ms_step / 2, 5),
                     "traffic": committed_traffic("block_copy.cu", "block_copy_cow.md")},
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_fused_write(args, dev, pa):
    """Diagnostic line for the q/k RMSNorm + rotary embedding fused into the KV write."""
    import numpy as np
    import torch
    rank, world, _ = dist_env()
    layers, T, hq, hkv, nb, max_pos = 28, 2048, 16, 8, 512, 4096
    g = torch.Generator(device=dev).manual_seed(11)
    bf = torch.bfloat16
    ins = [dict(q=torch.randn((T, hq, 128), generator=g, device=dev).to(bf),
                k=torch.randn((T, hkv, 128), generator=g, device=dev).to(bf),
                v=torch.randn((T, hkv, 128), generator=g, device=dev).to(bf),
                wq=(1 + 0.1 * torch.randn(128, generator=g, device=dev)).to(bf),
                wk=(1 + 0.1 * torch.randn(128, generator=g, device=dev)).to(bf),
                kc=torch.zeros((nb, 16, hkv, 128), device=dev, dtype=bf),
                vc=torch.zeros((nb, 16, hkv, 128), device=dev, dtype=bf)) for _ in range(layers)]
    q_out = [torch.empty_like(x["q"]) for x in ins]
    inv = 1.0 / (1e6 ** (torch.arange(0, 128, 2, dtype=torch.float32) / 128))
    f = torch.outer(torch.arange(max_pos, dtype=torch.float32), inv)
    cos = torch.cat([f.cos(), f.cos()], -1).to(bf).to(dev)
    sin = torch.cat([f.sin(), f.sin()], -1).to(bf).to(dev)
    rng = np.random.default_rng(11)
    pos = torch.from_numpy(np.concatenate([np.arange(0, 512), np.arange(512, 1024), np.arange(1536, 2048),
                                           rng.integers(16, 1024, size=512)]).astype(np.int32)).to(dev)
    slots = torch.from_numpy(rng.permutation(nb * 16)[:T].astype(np.int64)).to(dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        for l, x in enumerate(ins):
            pa.qk_norm_rope_kv_write(x["q"], x["k"], x["v"], x["wq"], x["wk"], 1e-6, cos, sin, pos, slots,
                                     x["kc"], x["vc"], q_out=q_out[l])

    g_step = graph_of(step, 1, stream)
    _device_error_check(pa)
    time_replays(g_step, max(args.warmup, 3), stream)
    barrier(dev)
    torch.cuda.synchronize()
    with ClockSampler(ClockSampler.gpu_id(dev)) as clk:
        reps = timed_repeats(lambda: time_replays(g_step, args.steps, stream), args.min_seconds)
        ms_step = statistics.median(reps) / args.steps
    ms_step = reduce_max(ms_step, dev)
    _device_error_check(pa)
    hbm, _, peak_kind = measured_peaks()
    # q read + q_out written, k and v read + written into the pool, each token's cos and sin rows read
    launch_bytes = T * (2 * hq * 256 + 4 * hkv * 256 + 2 * 256)
    gbs = layers * launch_bytes / (ms_step * 1e-3) / 1e9
    line = {
        "metric": "q/k RMSNorm + RoPE + KV write GB/s", "value": round(world * gbs, 1), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{T} new tokens per layer (chunks of 512 at prefixes 0, 512, 1536 + 512 decode "
                               f"tokens), Hq={hq}, Hkv={hkv}, d=128, bf16, {layers} layers with their own inputs "
                               f"and pools, rotary tables of {max_pos} positions (theta 1e6)",
                   "l2": f"{layers} layers x {launch_bytes / 1e6:.1f} MB of distinct inputs and outputs per step",
                   "timing": "CUDA events around a CUDA graph of one step, replayed K times"},
        "gpu_launches": layers * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs / hbm, 3), "peak_kind": peak_kind, "kernel": "qk_norm_rope_kv_write",
                     "bytes_per_launch": launch_bytes, "launch_ms": round(ms_step / layers, 5),
                     "traffic": committed_traffic("rope_write.cu", "rope_write_fused_write.md")},
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args):
    """The reference arm: the fp64 oracle (the pages print no runnable
    implementation of this path) timed on the host cores on the default
    line's workload, one decode layer call of the Qwen3-8B step per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import workloads
    oracle.build()
    case = workloads.qwen3_8b_decode(device="cpu", n_layers=1, nan_fill=False)
    threads = os.cpu_count() or 1
    kh, vh, qh = _u16(case.k_cache[0]), _u16(case.v_cache[0]), _u16(case.q[0])
    bt, ctx = case.block_tables.numpy(), case.context_lens.numpy()
    lay_bytes = workloads.decode_kv_bytes(case.meta["decode_lens"], case.hkv)
    for _ in range(max(args.warmup, 1)):
        oracle.paged_attn_decode(qh, kh, vh, bt, ctx, case.scale, oracle.BF16, num_threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.paged_attn_decode(qh, kh, vh, bt, ctx, case.scale, oracle.BF16, num_threads=threads)
    dt = time.perf_counter() - t0
    ms_step = dt * 1e3 / args.steps
    value = lay_bytes / (dt / args.steps) / 1e9
    sample = f"1 of the 36 decode layers of the Qwen3-8B step per step (fp64 C oracle, {threads} threads)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS[4][0], "global_batch": 64, "seq_len": case.max_context_len,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
