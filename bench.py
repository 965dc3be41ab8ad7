"""Benchmark of the MoE dispatch + combine hot path on GB300.

One step = moe_layout + moe_dispatch + moe_combine (TOPK_RANKS: the top-k
weighted reduction grouped by rank and the cross-rank sum) over one batch of
synthetic input, through the C ABI. Default workload: prefill, N=4096 tokens,
hidden 7168 BF16 ~N(0,1), 256 experts in 8 groups (top-4 groups, top-8
experts), R=8 virtual ranks, FP8 e4m3 per-128 dispatch, BF16 combine. Expert
outputs come from an identity expert (the dequantised records), made once
before timing: the expert itself is not part of the path.

Prints one JSON line. `--impl reference` times the plain CPU oracle instead
(rank 0 only), on bounded samples of the same workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload prefill|decode|decode_ll|rs|skewed|tiny|...]
Multi-GPU runs (torchrun) are independent replicas: the path has no
cross-GPU exchange on one-GPU-per-rank hardware here.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s and HBM GB/s vs GB300 roofline (1 GPU)"
L2_FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------- workloads --

def workload_spec(name: str) -> dict:
    """Shapes and algorithmic bytes per token for each kernel of a step."""
    if name == "prefill":
        s = dict(num_tokens=4096, hidden=7168, num_experts=256, topk=8, num_ranks=8,
                 out_kind="fp8", record_bytes=7472,
                 text="prefill N=4096 H=7168 E=256 (8 groups, top-4 groups) top-8 R=8; "
                      "FP8 e4m3 per-128 dispatch; BF16 combine grouped by rank")
    elif name == "skewed":
        s = dict(num_tokens=16384, hidden=7168, num_experts=256, topk=8, num_ranks=16,
                 out_kind="fp8", record_bytes=7472,
                 text="skewed N=16384 H=7168 E=256 Zipf(1.2) top-8 R=16; FP8 dispatch; "
                      "BF16 combine grouped by rank")
    elif name == "decode":
        s = dict(num_tokens=256, hidden=7168, num_experts=256, topk=8, num_ranks=8,
                 out_kind="raw", record_bytes=4112,
                 text="decode N=256 top-8 of 256 R=8; raw NVFP4 payload 3584 B + 448 B "
                      "scales per token; BF16 combine H=7168 grouped by rank")
    elif name == "rs":
        s = dict(num_tokens=2048, hidden=8192, num_experts=256, topk=8, num_ranks=4,
                 out_kind="bf16", record_bytes=16 + 32 + 32 + 16384,
                 text="reduce-scatter workload R=4 H=8192 512 tokens/rank (8 MiB/rank); "
                      "BF16 dispatch; top-8 of 256 combine grouped by rank")
    elif name == "prefill_norm":
        s = dict(num_tokens=4096, hidden=7168, num_experts=256, topk=8, num_ranks=8,
                 out_kind="fp8", record_bytes=7472, norm=True,
                 text="prefill N=4096 H=7168 E=256 top-8 R=8; FP8 dispatch; BF16 combine "
                      "grouped by rank fused with residual add and RMSNorm")
    elif name == "prefill_ranks":
        s = dict(num_tokens=4096, hidden=7168, num_experts=256, topk=8, num_ranks=8,
                 out_kind="fp8", record_bytes=7472, per_rank=True,
                 text="prefill N=4096 H=7168 E=256 top-8 R=8; one record per (token, rank) "
                      "(FP8 dispatch), rank rows summed back (BF16 combine)")
    elif name == "prefill_bwd":
        s = dict(num_tokens=4096, hidden=7168, num_experts=256, topk=8, num_ranks=8,
                 out_kind="fp8", record_bytes=7472, bwd=True,
                 names=("handle", "combine_backward", "dispatch_backward"),
                 text="prefill backward N=4096 H=7168 E=256 top-8 R=8: with the forward's slot "
                      "map cached, combine backward (bf16(w*g) to each pair's row and the fp32 "
                      "weight gradient) then dispatch backward (sum of each token's k rows)")
    elif name == "decode_ll":
        s = dict(num_tokens=1024, hidden=7168, num_experts=256, topk=8, num_ranks=8,
                 out_kind="fp8", record_bytes=7472, ll=True, max_tokens_per_rank=128,
                 text="low-latency decode: 8 ranks x 128 tokens, H=7168, top-8 of 256 experts; "
                      "FP8 e4m3 per-128 into fixed-capacity expert-major buffers "
                      "[256 x 1024 positions]; BF16 top-k combine")
    elif name == "tiny":
        s = dict(num_tokens=128, hidden=1024, num_experts=16, topk=2, num_ranks=2,
                 out_kind="bf16", record_bytes=2096,
                 text="tiny N=128 H=1024 E=16 top-2 R=2; BF16 dispatch and combine")
    else:
        raise SystemExit(f"unknown workload {name}")
    n, h, k, r = s["num_tokens"], s["hidden"], s["topk"], s["num_ranks"]
    in_row = 3584 + 448 if s["out_kind"] == "raw" else 2 * h
    # Algorithmic bytes per token: what each step must move at least once.
    s["bytes_per_token"] = dict(
        layout=4 * k + 4 * k + 4 * k + r,                     # ids in; slot_of, src_of_slot, mask out
        dispatch=in_row + 4 * k + 4 * k + 4 * k + k * s["record_bytes"],  # row, ids, w, slots in; k records out
        combine=k * 2 * h + 4 * k * 3 + 2 * h,                # k expert rows, w, slots, ids in; row out
    )
    if s.get("norm"):  # + residual in, normed and new residual out
        s["bytes_per_token"]["combine"] += 2 * 2 * h
    if s.get("bwd"):
        s["bytes_per_token"] = dict(
            layout=0,                                          # the cached slot map: no work
            dispatch=2 * h + 8 * k + k * 2 * h * 2 + 4 * k,    # g, w, slots, k rows of y in; k rows, grad_w out
            combine=k * 2 * h + 4 * k + 2 * h,                 # k gradient rows, slots in; row out
        )
    if s.get("ll"):
        e = s["num_experts"]
        cap = r * s["max_tokens_per_rank"]
        s["bytes_per_token"] = dict(
            # moe_layout as above + ll_slot_of out, and the whole src_info
            # [E, cap], layout_range [E, R] and recv_count [E] written
            layout=4 * k + 4 * k + 4 * k + r + 4 * k + (4 * e * cap + 8 * e * r + 4 * e) / n,
            # row, slots in; k payload rows + k scale rows out
            dispatch=2 * h + 4 * k + k * (h + 4 * (h // 128)),
            # k expert rows, weights, slots in; row out
            combine=k * 2 * h + 4 * k * 2 + 2 * h,
        )
    s["name"] = name
    return s


def make_inputs(spec: dict, seed: int = 0) -> dict:
    from combine_moe_layout_03_gb300 import synth
    n = spec["num_tokens"]
    if spec["name"] in ("prefill", "prefill_norm", "prefill_ranks", "prefill_bwd"):
        return synth.prefill_case(seed=seed, n=n)
    if spec["name"] == "skewed":
        return synth.skewed_case(seed=seed, n=n)
    if spec["name"] == "decode_ll":
        return synth.decode_ll_case(seed=seed, tokens_per_rank=spec["max_tokens_per_rank"],
                                    r=spec["num_ranks"])
    if spec["name"] == "decode":
        return synth.decode_case(seed=seed, n=n)
    if spec["name"] == "rs":
        c = synth.rs_case(seed=seed, tokens_per_rank=n // 4, with_partials=False,
                          with_expert_out=False)
        c["hidden_bf16"] = synth.bf16_normal(synth.rng_for(seed, 9), (n, spec["hidden"]))
        return c
    return synth.tiny_case(seed=seed)


# ---------------------------------------------------------------- clocks -----

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.lines = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [[x.strip() for x in line.split(",")] for line in out.splitlines() if line.strip()]
        rows = [r for r in rows if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = [v for v in sm if smax and v >= 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


def gpu_uuid():
    try:
        import torch
        u = str(torch.cuda.get_device_properties(0).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------- peaks ------

def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def recorded_traffic(kernel: str, workload: str) -> int | None:
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's source file changed since the counters were taken (each line
    names the .cu file and its hash at capture time)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        if line.startswith("#") or "=" not in line:
            continue
        kv = dict(x.split("=", 1) for x in line.split())
        if kv.get("kernel") != kernel or kv.get("workload") != workload:
            continue
        src = os.path.join(ROOT, "combine_moe_layout_03_gb300", "csrc", kv.get("source", ""))
        if not kv.get("source") or not os.path.exists(src):
            return None
        with open(src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
        return int(kv["bytes_per_launch"]) if kv.get("source_sha256") == sha else None
    return None


# ---------------------------------------------------------------- our arm ----

def layout_launches(n: int, k: int, e: int, r: int) -> int:
    """Kernels moe_layout launches: one cluster launch while the ids of a
    cluster block (up to 16 blocks of ~2048 pairs) and its histograms fit in
    200 KB of shared memory, else two (count, assign). Mirrors layout.cu."""
    pairs = n * k
    per = min(max(pairs // 16, 256), 2048)
    g = min(max(-(-pairs // per), 1), 16)
    tpb = -(-n // g)
    tpb = (tpb + 3) // 4 * 4
    smem = (36 + 3 * e + r + 1 + 16 * e) * 4 + tpb * k * 4
    return 1 if smem <= 200 * 1024 else 2


def single_kernel_layout_dispatch(n: int, k: int, e: int) -> bool:
    """Whether moe_layout_dispatch runs as one kernel: a routing of at most
    2048 pairs, or of MOE_FUSED_LAYOUT=p pairs (at most 2048; 0 turns it off).
    Mirrors dispatch.cu; the shared-memory bound there holds for every
    workload here."""
    v = os.environ.get("MOE_FUSED_LAYOUT")
    try:
        limit = 2048 if not v else min(max(int(v), 0), 2048)
    except ValueError:
        limit = 0
    return 0 < n * k <= limit and e <= 1024


class Step:
    """Resident buffers and the three calls of one step."""

    def __init__(self, spec: dict, dev, seed: int = 0):
        import torch
        from combine_moe_layout_03_gb300 import moe
        self.moe = moe
        self.spec = spec
        c = make_inputs(spec, seed)
        n, k, e, r, h = (spec["num_tokens"], spec["topk"], spec["num_experts"],
                         spec["num_ranks"], spec["hidden"])
        self.host = c
        # the step's inputs (ids, weights, the row, raw scales) as 256-byte-
        # aligned views of one device buffer, so that a step's host copy is a
        # single transfer (the end-to-end measurement)
        if spec["out_kind"] == "raw":
            parts = [c["topk_idx"], c["topk_weights"], c["payload"], c["scales"]]
        else:
            parts = [c["topk_idx"], c["topk_weights"], c["hidden_bf16"].view(np.int16)]
        offs, total = [], 0
        for a in parts:
            offs.append(total)
            total += (a.nbytes + 255) // 256 * 256
        staged = np.zeros(total, np.uint8)
        for a, o in zip(parts, offs):
            staged[o:o + a.nbytes] = np.ascontiguousarray(a).reshape(-1).view(np.uint8)
        self.inputs = torch.from_numpy(staged).to(dev)

        def view(i, dtype):
            a = parts[i]
            return self.inputs[offs[i]:offs[i] + a.nbytes].view(dtype).view(a.shape)

        self.ids = view(0, torch.int32)
        self.w = view(1, torch.float32)
        if spec["out_kind"] == "raw":
            self.x = view(2, torch.uint8)
            self.sc = view(3, torch.uint8)
            self.desc = moe.MoeDesc(n, k, e, r, h, moe.MOE_PAYLOAD_RAW, moe.MOE_PAYLOAD_RAW,
                                    3584, 448)
        else:
            self.x = view(2, torch.bfloat16)
            self.sc = None
            kind = moe.MOE_PAYLOAD_FP8_E4M3_B128 if spec["out_kind"] == "fp8" else moe.MOE_PAYLOAD_BF16
            self.desc = moe.MoeDesc(n, k, e, r, h, moe.MOE_PAYLOAD_BF16, kind)
        self.cdesc = moe.MoeDesc(n, k, e, r, h)
        # the rank-grouped combine needs whole ranks of tokens
        self.combine_mode = moe.MOE_COMBINE_TOPK_RANKS if n % r == 0 else moe.MOE_COMBINE_TOPK
        self.lay = moe.layout_outputs(self.desc, dev)
        self.ws = torch.empty(max(moe.moe_workspace_size(self.desc), 256), dtype=torch.uint8,
                              device=dev)
        rl = moe.moe_record_layout(self.desc)
        assert rl["record_bytes"] == spec["record_bytes"]
        self.records = torch.empty((n * k, rl["record_bytes"]), dtype=torch.uint8, device=dev)
        self.out = torch.empty((n, h), dtype=torch.bfloat16, device=dev)
        # identity expert, once: the records' payload back to BF16 rows
        moe.moe_layout(self.desc, self.ids, self.lay, self.ws)
        moe.moe_dispatch(self.desc, self.ids, self.w, self.x, self.sc, self.lay["slot_of"],
                         self.records)
        torch.cuda.synchronize()
        if spec["out_kind"] == "fp8":
            q = self.records[:, rl["off_payload"]:rl["off_payload"] + h].contiguous()
            s = self.records[:, rl["off_scales"]:rl["off_scales"] + 4 * (h // 128)].contiguous()
            self.y = (q.view(torch.float8_e4m3fn).float()
                      * s.view(torch.float32).repeat_interleave(128, dim=1)).to(torch.bfloat16)
        elif spec["out_kind"] == "bf16":
            self.y = self.records[:, rl["off_payload"]:rl["off_payload"] + 2 * h].contiguous() \
                .view(torch.bfloat16)
        else:  # raw NVFP4 bytes: the expert's output rows are drawn directly
            from combine_moe_layout_03_gb300 import synth
            yy = synth.bf16_normal(synth.rng_for(seed, 11), (n * k, h))
            self.y = torch.from_numpy(yy.view(np.int16)).to(dev).view(torch.bfloat16)
        self.launches_per_step = layout_launches(n, k, e, r) + 1 + 1
        if spec.get("ll"):
            self._setup_ll(spec, dev)
            return
        if spec.get("bwd"):
            self._setup_bwd(spec, dev, seed)
            return
        if spec.get("per_rank"):
            self._setup_per_rank(spec, dev, seed)
            return
        # the three calls with their arguments marshalled once (same buffers
        # every step), so host overhead stays well below the GPU's step time
        self.layout = moe.prepare_layout(self.desc, self.ids, self.lay, self.ws)
        self.dispatch = moe.prepare_dispatch(self.desc, self.ids, self.w, self.x, self.sc,
                                             self.lay["slot_of"], self.records)
        # the step itself runs layout and dispatch as one call, whose dispatch
        # overlaps the layout (the breakdown loop times the two separately)
        self.layout_dispatch = moe.prepare_layout_dispatch(self.desc, self.ids, self.w, self.x, self.sc,
                                                           self.lay, self.ws, self.records)
        if single_kernel_layout_dispatch(n, k, e):
            self.launches_per_step = 1 + 1
        if spec.get("norm"):
            from combine_moe_layout_03_gb300 import synth
            self.residual = torch.from_numpy(synth.bf16_normal(synth.rng_for(seed, 12), (n, h))
                                             .view(np.int16)).to(dev).view(torch.bfloat16)
            self.gamma = torch.from_numpy(synth.bf16_normal(synth.rng_for(seed, 13), (h,))
                                          .view(np.int16)).to(dev).view(torch.bfloat16)
            self.residual_out = torch.empty_like(self.out)
            self.combine = moe.prepare_combine_norm(
                self.cdesc, moe.MOE_COMBINE_TOPK_RANKS, self.y, self.ids, self.w,
                self.lay["slot_of"], self.residual, self.gamma, 1e-6, self.out, self.residual_out)
        else:
            self.combine = moe.prepare_combine(self.cdesc, self.combine_mode, self.y,
                                               self.ids, self.w, self.lay["slot_of"], self.out)

    def _setup_per_rank(self, spec, dev, seed):
        """One record per (token, rank): the layout and the receive layout in
        one call (moe_layout_ranks, timed as 'layout'); the expert of rank r
        returns, per received token, the sum of its local pairs' weight times
        the dequantised row."""
        import torch
        moe = self.moe
        n, h = spec["num_tokens"], spec["hidden"]
        self.rlay = moe.moe_rank_layout(self.desc, self.lay)
        recv = int(self.rlay["recv_offset"][-1].item())
        self.records = torch.empty((n * spec["num_ranks"], spec["record_bytes"]), dtype=torch.uint8,
                                   device=dev)
        moe.moe_dispatch_ranks(self.desc, self.ids, self.w, self.x, self.sc,
                               self.rlay["send_head"], self.records)
        torch.cuda.synchronize()
        rl = moe.moe_record_layout(self.desc)
        rec = self.records[:recv]
        q = rec[:, rl["off_payload"]:rl["off_payload"] + h].contiguous().view(torch.float8_e4m3fn)
        sc = rec[:, rl["off_scales"]:rl["off_scales"] + 4 * (h // 128)].contiguous().view(torch.float32)
        lw = rec[:, rl["off_weights"]:rl["off_weights"] + 4 * spec["topk"]].contiguous().view(torch.float32)
        self.y = (q.float() * sc.repeat_interleave(128, dim=1) * lw.sum(1, keepdim=True)).to(torch.bfloat16)
        self.recv_records = recv
        import torch
        self.layout, self.dispatch, self.combine = self._rank_calls_on(torch.cuda.current_stream())
        # the receive layout runs inside the cluster layout launch, or as a
        # third kernel after the two-kernel layout
        nl = layout_launches(n, spec["topk"], spec["num_experts"], spec["num_ranks"])
        self.launches_per_step = nl + (0 if nl == 1 else 1) + 1 + 1
        # algorithmic bytes per token from the actual (token, rank) records
        per = recv / n
        r = spec["num_ranks"]
        spec["bytes_per_token"] = dict(
            layout=12 * spec["topk"] + r + r + 4 * r + 4 * r,  # + mask in, send_head, recv_src_idx out
            dispatch=2 * h + 12 * spec["topk"] + 4 * r + per * spec["record_bytes"],
            combine=per * 2 * h + 4 * r + 2 * h,
        )

    def _setup_ll(self, spec, dev):
        """Fixed-capacity, expert-major buffers: the layout and the fixed-capacity
        layout in one call (moe_layout_ll, timed as 'layout'), the payload and scales go to
        [E * capacity] rows, and the expert of each position returns its
        dequantised row; the combine is the top-k reduction over those rows."""
        import torch
        moe = self.moe
        h, max_t = spec["hidden"], spec["max_tokens_per_rank"]
        self.ll = moe.moe_ll_layout(self.desc, max_t, self.ids, self.lay)
        cap = self.ll["capacity"]
        rows = spec["num_experts"] * cap
        rl = moe.moe_record_layout(self.desc)
        self.x_ll = torch.empty((rows, rl["payload_bytes"]), dtype=torch.uint8, device=dev)
        self.s_ll = torch.empty((rows, rl["scale_bytes"]), dtype=torch.uint8, device=dev)
        moe.moe_dispatch_ll(self.desc, self.x, self.sc, self.ll["ll_slot_of"], cap, self.x_ll,
                            self.s_ll)
        torch.cuda.synchronize()
        pos = self.ll["ll_slot_of"].flatten()
        pos = pos[pos >= 0].long()
        q = self.x_ll.index_select(0, pos).view(torch.float8_e4m3fn)
        sc = self.s_ll.index_select(0, pos).contiguous().view(torch.float32)
        self.records = None
        self.y = torch.zeros((rows, h), dtype=torch.bfloat16, device=dev)
        self.y[pos] = (q.float() * sc.repeat_interleave(128, dim=1)).to(torch.bfloat16)
        self.max_t = max_t
        self.calls_on = self._ll_calls_on
        h = torch.cuda.current_stream().cuda_stream
        self.layout = moe.prepare_layout_ll(self.desc, self.max_t, self.ids, self.lay, self.ll, self.ws, h)
        self.dispatch = moe.prepare_dispatch_ll(self.desc, self.x, self.sc, self.ll["ll_slot_of"],
                                                self.x_ll, self.s_ll, h)
        # the step runs layout and dispatch as one call (the breakdown times
        # them apart)
        self.layout_dispatch, self.combine = self._ll_calls_on(torch.cuda.current_stream())
        # the fixed-capacity layout runs inside the cluster layout launch (this
        # workload's source ranks are whole blocks), or after the two-kernel one
        nl = layout_launches(spec["num_tokens"], spec["topk"], spec["num_experts"], spec["num_ranks"])
        self.launches_per_step = nl + (0 if nl == 1 else 1) + 2

    def _setup_bwd(self, spec, dev, seed):
        """The backward step with the forward's slot map cached: the upstream
        gradient g (in the role of the step's input) goes through combine
        backward into the pairs' gradient rows and weight gradients, and
        dispatch backward sums each token's rows into grad_hidden (the step's
        output)."""
        import torch
        from combine_moe_layout_03_gb300 import synth
        moe = self.moe
        n, k, h = spec["num_tokens"], spec["topk"], spec["hidden"]
        P = self.y.shape[0]
        # g goes into the packed input buffer in place of the row
        self.x.copy_(torch.from_numpy(synth.bf16_normal(synth.rng_for(seed, 14), (n, h))
                                      .view(np.int16)).to(dev).view(torch.bfloat16))
        self.sc = None
        self.records = None
        self.grad_y = torch.empty((P, h), dtype=torch.bfloat16, device=dev)
        self.grad_w = torch.empty((n, k), dtype=torch.float32, device=dev)
        self.calls_on = self._bwd_calls_on
        cb, db = self._bwd_calls_on(torch.cuda.current_stream())
        self.layout = lambda: None
        self.dispatch, self.combine = cb, db
        self.launches_per_step = 2

    def _bwd_calls_on(self, stream):
        moe = self.moe
        h = stream.cuda_stream
        return [moe.prepare_combine_backward(self.cdesc, self.x, self.w, self.lay["slot_of"], self.y,
                                             self.y.shape[0], self.grad_y, self.grad_w, h),
                moe.prepare_dispatch_backward(self.cdesc, self.grad_y, self.lay["slot_of"],
                                              self.out, h)]

    def _ll_calls_on(self, stream):
        moe = self.moe
        h = stream.cuda_stream
        return [moe.prepare_layout_ll_dispatch(self.desc, self.max_t, self.ids, self.x, self.sc, self.lay,
                                               self.ll, self.ws, self.x_ll, self.s_ll, h),
                moe.prepare_combine(self.cdesc, moe.MOE_COMBINE_TOPK, self.y, self.ids, self.w,
                                    self.ll["ll_slot_of"], self.out, h)]

    def _rank_calls_on(self, stream):
        moe = self.moe
        h = stream.cuda_stream
        return [moe.prepare_layout_ranks(self.desc, self.ids, 1, self.lay, self.rlay, self.ws, h),
                moe.prepare_dispatch_ranks(self.desc, self.ids, self.w, self.x, self.sc,
                                           self.rlay["send_head"], self.records, h),
                moe.prepare_combine_gather_ranks(self.cdesc, self.y, self.rlay["send_head"],
                                                 self.out, h)]

    def run(self):
        fused = getattr(self, "layout_dispatch", None)
        if fused is not None:
            fused()
        else:
            self.layout()
            self.dispatch()
        self.combine()

    def calls_on(self, stream):
        """The step's three calls bound to `stream` (for graph capture)."""
        moe = self.moe
        h = stream.cuda_stream
        if self.spec.get("per_rank"):
            return self._rank_calls_on(stream)
        calls = [moe.prepare_layout_dispatch(self.desc, self.ids, self.w, self.x, self.sc, self.lay,
                                             self.ws, self.records, h)]
        if self.spec.get("norm"):
            calls.append(moe.prepare_combine_norm(
                self.cdesc, moe.MOE_COMBINE_TOPK_RANKS, self.y, self.ids, self.w,
                self.lay["slot_of"], self.residual, self.gamma, 1e-6, self.out,
                self.residual_out, h))
        else:
            calls.append(moe.prepare_combine(self.cdesc, self.combine_mode, self.y,
                                             self.ids, self.w, self.lay["slot_of"], self.out, h))
        return calls


def measure_graph(st: "Step", K: int, flush, flush_read) -> dict:
    """The whole step captured once in a CUDA graph and replayed: device time
    per replay (CUDA events around each replay, L2 flushed in between)."""
    import torch
    s = torch.cuda.Stream()
    calls = st.calls_on(s)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            for c in calls:
                c()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for c in calls:
            c()
    k2 = max(3, min(K, 200))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(k2)]
    for _ in range(3):
        g.replay()
    for a, b in ev:
        flush.zero_()
        flush_read.sum()
        a.record()
        g.replay()
        b.record()
    torch.cuda.synchronize()
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in ev)
    return {"step_us_median": round(us[len(us) // 2], 2), "step_us_min": round(us[0], 2),
            "replays": k2}


def run_ag_slots(args, rank, world):
    """The decode all-gather's data path on one GPU: mask padded tokens, pack
    8 ranks x 256 tokens of (ids, weights, NVFP4 payload, scales) into
    16-byte-aligned rank slots, and unpack them into the gathered tensors."""
    import torch
    from combine_moe_layout_03_gb300 import moe, synth
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    r, n = 8, 256
    c = synth.decode_case(seed=rank, n=r * n)
    ts = [torch.from_numpy(np.ascontiguousarray(c[key])).to(dev)
          for key in ("topk_idx", "topk_weights", "payload", "scales")]
    n_act = torch.tensor([r * n - 3], dtype=torch.int32, device=dev)
    slots = moe.moe_pack_slots(ts, r)
    outs = [torch.empty_like(t) for t in ts]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_read = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    K, W = args.steps, args.warmup
    for _ in range(W):
        moe.moe_mask_topk_ids(ts[0], n_act)
        moe.moe_pack_slots(ts, r, slots)
        moe.moe_unpack_slots(slots, outs, r)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    torch.cuda.synchronize()
    for i in range(K):
        flush.zero_()
        flush_read.sum()
        ev[i][0].record()
        moe.moe_mask_topk_ids(ts[0], n_act)
        ev[i][1].record()
        moe.moe_pack_slots(ts, r, slots)
        ev[i][2].record()
        moe.moe_unpack_slots(slots, outs, r)
        ev[i][3].record()
    torch.cuda.synchronize()
    per = {name: statistics.mean(ev[i][a].elapsed_time(ev[i][b]) for i in range(K))
           for name, a, b in (("mask", 0, 1), ("pack", 1, 2), ("unpack", 2, 3))}
    total_ms, value = whole_job(sum(ev[i][0].elapsed_time(ev[i][3]) for i in range(K)),
                                r * n * K, world, dev)
    slot_bytes = slots.numel()
    peak = measured_peaks()
    gbs = {name: 2 * slot_bytes / (per[name] / 1e3) / 1e9 for name in ("pack", "unpack")}
    return {
        "metric": "decode all-gather slot packing tokens/s and HBM GB/s", "value": round(value, 1),
        "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(total_ms / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bytes", "data": "synthetic",
        "config": {"workload": "decode all-gather payload: 8 ranks x 256 tokens, top-8 ids and "
                               "weights, 3584 B NVFP4 + 448 B scales per token; mask, pack, unpack",
                   "slot_bytes_per_rank": slot_bytes // r},
        "kernels_us": {k: round(v * 1e3, 2) for k, v in per.items()},
        "kernels_gbs": {k: round(v, 1) for k, v in gbs.items()},
        "kernels_frac": {k: round(v / peak["hbm_gbs"], 4) for k, v in gbs.items()},
        "gpu_launches": 3 * K,
    }


def _timed(fn, K, flush, flush_read, stream):
    """Mean device time of fn over K calls (CUDA events at its ends, L2
    flushed before each call), in microseconds."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev:
        flush.zero_()
        flush_read.sum()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3


def _timed_b2b(fns, K, stream):
    """Mean device time per call of K calls issued back to back (the pages'
    method: events around many repeats), cycling through fns, which work on
    separate buffer copies whose total exceeds L2 so that every call reads
    from DRAM; in microseconds."""
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for i in range(K):
        fns[i % len(fns)]()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / K


DECODE_SWEEP_N = (1, 2, 4, 8, 16, 32, 64, 128, 256)
RS_SWEEP_T = (32, 64, 128, 256, 512)


def decode_sweep_rows(dev, K, W, seed_base, flush, flush_read, stream):
    """The decode step at each N of DECODE_SWEEP_N: eager step time (events at
    the step's ends, L2 flushed before each step) and CUDA-graph replay time.
    Returns (rows, kernels launched, eager ms in total, tokens in total)."""
    rows, launches, total_ms, total_tokens = [], 0, 0.0, 0
    for n in DECODE_SWEEP_N:
        spec = workload_spec("decode")
        spec["num_tokens"] = n
        st = Step(spec, dev, seed=seed_base + n)
        for _ in range(W):
            st.run()
        eager = _timed(st.run, K, flush, flush_read, stream)
        graph = measure_graph(st, K, flush, flush_read)
        rows.append({"num_tokens": n, "eager_step_us": round(eager, 2),
                     "graph_step_us": graph["step_us_median"],
                     "graph_tokens_per_s": round(n / (graph["step_us_median"] / 1e6), 1)})
        launches += st.launches_per_step * (K + graph["replays"])
        total_ms += eager * K / 1e3
        total_tokens += n * K
        del st
    return rows, launches, total_ms, total_tokens


def run_decode_sweep(args, rank, world):
    """The decode step at N = 1, 2, 4, ..., 256 tokens (raw NVFP4 payload,
    top-8 of 256, R=8; the combine grouped by rank where N % R == 0): eager
    step time and CUDA-graph replay time per N."""
    import torch
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_read = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    K, W = min(args.steps, 100), args.warmup
    clocks = ClockSampler(gpu_uuid())
    rows, launches, total_ms, total_tokens = decode_sweep_rows(dev, K, W, rank * 1000, flush,
                                                               flush_read, stream)
    clk = clocks.stop()
    total_ms, value = whole_job(total_ms, total_tokens, world, dev)
    last = rows[-1]
    return {
        "metric": METRIC, "value": round(last["num_tokens"] / (last["eager_step_us"] / 1e6), 1),
        "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(last["eager_step_us"] / 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "raw bytes (NVFP4 payload), bf16 combine",
        "data": "synthetic",
        "config": {"workload": "decode sweep: N = 1..256 tokens, top-8 of 256 R=8, raw 3584 B + 448 B "
                               "payload per token, BF16 combine H=7168 (value and ms_per_step at N=256)",
                   "l2": "flushed before every timed step"},
        "sweep": rows, "gpu_launches": launches, "clocks": clk,
    }


def rs_sweep_rows(dev, K, W, seed_base, flush, flush_read, stream):
    """The combine as a reduce-scatter, R=4, H=8192, at each T of RS_SWEEP_T
    tokens per rank: the rank sum of BF16 partials and the top-8 reduction
    grouped by rank, one call after an L2 flush and calls back to back on
    copies of the inputs beyond twice the L2. Returns (rows, kernels
    launched, floor): floor times the rank sum of one token per rank (80 KB
    moved) both ways, the fixed cost every call of the sweep carries."""
    import torch
    from combine_moe_layout_03_gb300 import moe, synth
    peak = measured_peaks()["hbm_gbs"]
    r, h, k, e = 4, 8192, 8, 256
    rows, launches = [], 0
    c = synth.rs_case(seed=seed_base, tokens_per_rank=1, hidden=h, r=r, e=e, k=k, with_expert_out=False)
    part = torch.from_numpy(c["partials_bf16"].view(np.int16)).to(dev).view(torch.bfloat16)
    outs = [torch.empty((r, h), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    tiny = [moe.prepare_combine(moe.MoeDesc(r, k, e, r, h), moe.MOE_COMBINE_RANKS, part, None, None,
                                None, o) for o in outs]
    for _ in range(W):
        tiny[0]()
    floor = {"rank_sum_us": round(_timed(tiny[0], K, flush, flush_read, stream), 2),
             "rank_sum_us_back_to_back": round(_timed_b2b(tiny, K, stream), 2),
             "what": "rank sum of one token per rank (80 KB moved): the fixed cost of a call"}
    launches += W + 2 * K
    del tiny, outs, part
    for t in RS_SWEEP_T:
        c = synth.rs_case(seed=seed_base + t, tokens_per_rank=t, hidden=h, r=r, e=e, k=k)
        n = r * t
        d = moe.MoeDesc(n, k, e, r, h)
        part = torch.from_numpy(c["partials_bf16"].view(np.int16)).to(dev).view(torch.bfloat16)
        y = torch.from_numpy(c["expert_out_bf16"].view(np.int16)).to(dev).view(torch.bfloat16)
        ids = torch.from_numpy(c["topk_idx"]).to(dev)
        w = torch.from_numpy(c["topk_weights"]).to(dev)
        lay = moe.moe_layout(d, ids)
        out = torch.empty((n, h), dtype=torch.bfloat16, device=dev)
        ranks = moe.prepare_combine(d, moe.MOE_COMBINE_RANKS, part, None, None, None, out)
        fused = moe.prepare_combine(d, moe.MOE_COMBINE_TOPK_RANKS, y, ids, w, lay["slot_of"], out)
        for _ in range(W):
            ranks()
            fused()
        us_r = _timed(ranks, K, flush, flush_read, stream)
        us_f = _timed(fused, K, flush, flush_read, stream)
        b_r = (r * n * h + n * h) * 2            # R partials in, the sum out
        b_f = (k * n * h + n * h) * 2 + 12 * k * n  # k rows in, the sum out, pair info
        # back to back over copies of the inputs and outputs that together
        # exceed twice the L2
        copies = max(2, -(-2 * L2_FLUSH_BYTES // min(b_r, b_f)))
        parts = [part] + [part.clone() for _ in range(copies - 1)]
        ys = [y] + [y.clone() for _ in range(copies - 1)]
        outs = [out] + [torch.empty_like(out) for _ in range(copies - 1)]
        ranks_b = [moe.prepare_combine(d, moe.MOE_COMBINE_RANKS, parts[i], None, None, None, outs[i])
                   for i in range(copies)]
        fused_b = [moe.prepare_combine(d, moe.MOE_COMBINE_TOPK_RANKS, ys[i], ids, w, lay["slot_of"], outs[i])
                   for i in range(copies)]
        for f in ranks_b + fused_b:
            f()
        us_rb = _timed_b2b(ranks_b, K, stream)
        us_fb = _timed_b2b(fused_b, K, stream)
        rows.append({"tokens_per_rank": t, "out_mib_per_rank": t * h * 2 / 2 ** 20,
                     "rank_sum_us": round(us_r, 2), "rank_sum_frac": round(b_r / us_r / 1e3 / peak, 3),
                     "topk_ranks_us": round(us_f, 2), "topk_ranks_frac": round(b_f / us_f / 1e3 / peak, 3),
                     "rank_sum_us_back_to_back": round(us_rb, 2),
                     "rank_sum_frac_back_to_back": round(b_r / us_rb / 1e3 / peak, 3),
                     "topk_ranks_us_back_to_back": round(us_fb, 2),
                     "topk_ranks_frac_back_to_back": round(b_f / us_fb / 1e3 / peak, 3)})
        del parts, ys, outs, ranks_b, fused_b
        launches += 4 * K
    return rows, launches, floor


def run_rs_sweep(args, rank, world):
    """The combine as a reduce-scatter, R=4 ranks, H=8192, 32..512 tokens per
    rank (0.5..8 MiB of output per rank): (i) the cross-rank sum of R BF16
    partials, (ii) the top-8 weighted reduction grouped by rank. Device time
    per call."""
    import torch
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_read = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    K, W = min(args.steps, 100), args.warmup
    clocks = ClockSampler(gpu_uuid())
    rows, launches, floor = rs_sweep_rows(dev, K, W, rank * 1000, flush, flush_read, stream)
    clk = clocks.stop()
    r = 4
    last = rows[-1]
    return {
        "metric": METRIC, "value": round(r * last["tokens_per_rank"] / (last["topk_ranks_us"] / 1e6), 1),
        "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(last["topk_ranks_us"] / 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in/out, fp32 accumulate",
        "data": "synthetic",
        "config": {"workload": "reduce-scatter sweep: R=4, H=8192, 32..512 tokens per rank; rank sum "
                               "of BF16 partials and top-8 weighted reduction grouped by rank "
                               "(value at 512 tokens per rank, grouped form)",
                   "l2": "flushed before every timed call; the back-to-back columns cycle through "
                         "copies of the inputs larger than twice the L2 instead"},
        "sweep": rows, "floor": floor, "gpu_launches": launches, "clocks": clk,
        "pages_context_us": {"0.5": [42.4, 35.6], "1": [43.1, 37.1], "2": [42.3, 37.4],
                             "4": [51.6, 43.5], "8": [84.8, 76.7],
                             "note": "NCCL symmetric reduce-scatter, staged and direct, 4 GPUs over "
                                     "NVLink: a collective across GPUs, context only"},
    }


def step_and_breakdown(st: "Step", K: int, flush, flush_read, stream) -> dict:
    """Mean device time of K steps (events at each step's ends only, L2
    flushed between steps) and of each of its three calls (a second loop
    with an event between calls), in microseconds."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush.zero_()
        flush_read.sum()
        ev[i][0].record(stream)
        st.run()
        ev[i][1].record(stream)
    eb = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for i in range(K):
        flush.zero_()
        flush_read.sum()
        e = eb[i]
        e[0].record(stream)
        st.layout()
        e[1].record(stream)
        st.dispatch()
        e[2].record(stream)
        st.combine()
        e[3].record(stream)
    torch.cuda.synchronize()
    out = {"step": statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3}
    for name, a, b in (("layout", 0, 1), ("dispatch", 1, 2), ("combine", 2, 3)):
        out[name] = statistics.mean(eb[i][a].elapsed_time(eb[i][b]) for i in range(K)) * 1e3
    return out


def run_configs(args, dev, flush, flush_read, stream) -> dict:
    """The other workloads of the pages, measured in the same run as the
    headline line with fewer steps each: tiny (step and graph replay), the
    decode sweep N = 1..256 (graph replay), the reduce-scatter sweep 0.5..8
    MiB per rank (both combine forms) and skewed (dispatch, combine, step)."""
    K, W = max(3, min(args.steps, 20)), args.warmup
    peak = measured_peaks()["hbm_gbs"]
    clocks = ClockSampler(gpu_uuid())
    t0 = time.perf_counter()
    out, launches = {}, 0

    st = Step(workload_spec("tiny"), dev, seed=101)
    for _ in range(W):
        st.run()
    eager = _timed(st.run, K, flush, flush_read, stream)
    graph = measure_graph(st, K, flush, flush_read)
    launches += st.launches_per_step * (K + graph["replays"])
    out["tiny"] = {"step_us": round(eager, 2), "graph_us": graph["step_us_median"],
                   "what": "N=128 H=1024 E=16 top-2 R=2, BF16 dispatch and combine"}
    del st

    rows, n_l, _, _ = decode_sweep_rows(dev, K, W, 200, flush, flush_read, stream)
    launches += n_l
    out["decode_sweep"] = {"num_tokens": [r["num_tokens"] for r in rows],
                           "graph_us": [r["graph_step_us"] for r in rows],
                           "eager_us": [r["eager_step_us"] for r in rows],
                           "what": "top-8 of 256, R=8, raw 3584 B + 448 B payload, BF16 combine "
                                   "H=7168; one step = layout + dispatch + combine"}

    rows, n_l, floor = rs_sweep_rows(dev, K, W, 300, flush, flush_read, stream)
    launches += n_l
    out["rs_sweep"] = {"out_mib_per_rank": [r["out_mib_per_rank"] for r in rows]}
    for key in ("rank_sum_us", "rank_sum_frac", "topk_ranks_us", "topk_ranks_frac",
                "rank_sum_us_back_to_back", "rank_sum_frac_back_to_back",
                "topk_ranks_us_back_to_back", "topk_ranks_frac_back_to_back"):
        out["rs_sweep"][key] = [r[key] for r in rows]
    out["rs_sweep"]["floor_us"] = [floor["rank_sum_us"], floor["rank_sum_us_back_to_back"]]
    out["rs_sweep"]["what"] = ("R=4, H=8192: rank sum of BF16 partials and top-8 reduction grouped "
                               "by rank; one call after an L2 flush, and calls back to back")

    spec = workload_spec("skewed")
    st = Step(spec, dev, seed=400)
    for _ in range(W):
        st.run()
    t = step_and_breakdown(st, K, flush, flush_read, stream)
    launches += st.launches_per_step * K + 3 * K
    n, bpt = spec["num_tokens"], spec["bytes_per_token"]
    sk = {"step_us": round(t["step"], 2), "layout_us": round(t["layout"], 2),
          "tokens_per_s": round(n / (t["step"] / 1e6), 1)}
    for name in ("dispatch", "combine"):
        gbs = bpt[name] * n / (t[name] / 1e6) / 1e9
        sk[f"{name}_us"] = round(t[name], 2)
        sk[f"{name}_gbs"] = round(gbs, 1)
        sk[f"{name}_frac"] = round(gbs / peak, 4)
    sk["routing"] = routing_stats(st.lay["tokens_per_expert"], st.lay["tokens_per_rank"])
    sk["what"] = spec["text"]
    out["skewed"] = sk
    del st

    out["steps_each"] = K
    out["gpu_launches"] = launches
    out["clocks"] = clocks.stop()
    out["wall_s"] = round(time.perf_counter() - t0, 1)
    out["l2"] = "flushed before every timed step or call, except the back-to-back columns"
    return out


def run_ours(args, spec, rank, world):
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    # S seeded input sets (routing, hidden rows, expert outputs); timed step i
    # runs on set i % S
    S = max(1, args.seeds)
    sets = [Step(spec, dev, seed=rank * 1000 + j) for j in range(S)]
    st = sets[0]
    stream = torch.cuda.current_stream()
    # L2 flush between steps: write a buffer larger than L2, then read another
    # one, so the written lines are evicted (and written back) before the
    # step's events start rather than during its first kernels
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_read = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    K, W = args.steps, args.warmup
    clocks = ClockSampler(gpu_uuid())
    for i in range(W):
        sets[i % S].run()
    # The timed steps: events at the start and the end of each step only, so
    # that consecutive kernels may overlap their launch (programmatic
    # dependent launch) as they do in an application.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(K):
        flush.zero_()                  # L2 flush, outside the timed events
        flush_read.sum()
        ev[i][0].record(stream)
        sets[i % S].run()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    step_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    # The per-kernel breakdown: the same steps with an event between calls
    # (which serialises them), for each kernel's own duration.
    eb = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for i in range(K):
        flush.zero_()
        flush_read.sum()
        e = eb[i]
        sx = sets[i % S]
        e[0].record(stream)
        sx.layout()
        e[1].record(stream)
        sx.dispatch()
        e[2].record(stream)
        sx.combine()
        e[3].record(stream)
    torch.cuda.synchronize()
    per = {name: [eb[i][a].elapsed_time(eb[i][b]) for i in range(K)]
           for name, a, b in (("layout", 0, 1), ("dispatch", 1, 2), ("combine", 2, 3))}
    serial_ms = statistics.mean(eb[i][0].elapsed_time(eb[i][3]) for i in range(K))
    n = spec["num_tokens"]
    total_ms, value = whole_job(sum(step_ms), n * K, world, dev)
    peaks = measured_peaks()
    kern = {name: statistics.mean(v) for name, v in per.items()}
    dom = max(("dispatch", "combine"), key=lambda x: kern[x])
    bpt = spec["bytes_per_token"]
    achieved = {name: bpt[name] * n / (kern[name] / 1e3) / 1e9 if kern[name] > 0 else 0.0
                for name in kern}
    step_bytes = sum(bpt.values()) * n
    # where layout and dispatch run as one kernel, that call alone as well
    single = None
    if getattr(st, "layout_dispatch", None) is not None and \
            single_kernel_layout_dispatch(n, spec["topk"], spec["num_experts"]):
        es = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for i in range(K):
            flush.zero_()
            flush_read.sum()
            es[i][0].record(stream)
            sets[i % S].layout_dispatch()
            es[i][1].record(stream)
        torch.cuda.synchronize()
        t1 = statistics.mean(es[i][0].elapsed_time(es[i][1]) for i in range(K))
        gbs = (bpt["layout"] + bpt["dispatch"]) * n / (t1 / 1e3) / 1e9
        single = {"kernel": "k_layout_dispatch_small", "us": round(t1 * 1e3, 2), "gbs": round(gbs, 1),
                  "frac": round(gbs / peaks["hbm_gbs"], 4),
                  "traffic": None if spec.get("tokens_overridden")
                  else recorded_traffic("layout_dispatch_small", spec["name"])}
    # the three timed calls under their own names (the backward step's are
    # the cached handle, combine backward and dispatch backward)
    label = dict(zip(("layout", "dispatch", "combine"),
                     spec.get("names", ("layout", "dispatch", "combine"))))

    per_seed = [statistics.mean(step_ms[i] for i in range(j, K, S)) * 1e3 for j in range(min(S, K))]
    graph = measure_graph(st, K, flush, flush_read)
    e2e = measure_e2e(st, spec, dev, K, W, seed=rank) if rank == 0 else None
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(total_ms / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in/out, fp32 accumulate, e4m3 records" if spec["out_kind"] == "fp8"
        else "bf16 in/out, fp32 accumulate",
        "data": "synthetic (seeded; shapes and distributions of the pages' workloads)",
        "config": {"workload": spec["text"], "num_tokens": n, "hidden": spec["hidden"],
                   "num_experts": spec["num_experts"], "topk": spec["topk"],
                   "num_ranks": spec["num_ranks"], "record_bytes": spec["record_bytes"],
                   "combine_mode": "TOPK_RANKS + residual + RMSNorm" if spec.get("norm")
                   else "rank rows gathered per token" if spec.get("per_rank")
                   else "TOPK over the fixed-capacity positions" if spec.get("ll")
                   else "backward of TOPK combine and of dispatch" if spec.get("bwd") else "TOPK_RANKS",
                   "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write, then "
                         f"{L2_FLUSH_BYTES >> 20} MiB read, outside the timed events); step "
                         f"working set {step_bytes / 1e6:.0f} MB",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": label[dom], "achieved": round(achieved[dom], 1),
                     "peak": peaks["hbm_gbs"], "peak_source": peaks["source"], "unit": "GB/s",
                     "frac": round(achieved[dom] / peaks["hbm_gbs"], 4),
                     "traffic": None if spec.get("tokens_overridden") else recorded_traffic(label[dom], spec["name"]),
                     "algorithmic_bytes_per_launch": bpt[dom] * n},
        "kernels_us": {label[name]: round(v * 1e3, 2) for name, v in kern.items()},
        "kernels_gbs": {label[name]: round(v, 1) for name, v in achieved.items()},
        "kernels_frac": {label[name]: round(v / peaks["hbm_gbs"], 4) for name, v in achieved.items()},
        "step_gbs": round(step_bytes / (total_ms / K / 1e3) / 1e9, 1),
        "ms_per_step_serialised": round(serial_ms, 5),
        "seeds": {"count": S, "step_us_per_seed": [round(x, 2) for x in per_seed],
                  "step_us_median": round(statistics.median(per_seed), 2)},
        "gpu_launches": st.launches_per_step * K,
        "pdl": os.environ.get("MOE_PDL", "1") != "0",
        "graph": graph,
        "clocks": clk,
        "wall_s": round(wall, 3),
    }
    if single is not None:
        line["layout_dispatch_one_kernel"] = single
    if e2e is not None:
        line["e2e"] = e2e
    if getattr(st, "lay", None) is not None and "tokens_per_expert" in st.lay:
        line["routing"] = routing_stats(st.lay["tokens_per_expert"], st.lay["tokens_per_rank"])
    if spec["name"] == "prefill" and not spec.get("tokens_overridden") and world == 1 \
            and not args.no_configs:
        del sets, st
        line["configs"] = run_configs(args, dev, flush, flush_read, stream)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, budget_s=args.cpu_seconds)
    return line


def routing_stats(tokens_per_expert, tokens_per_rank) -> dict:
    """Load balance of the first input set's routing, from the layout kernel's
    own outputs (read once, after the timed steps): pairs per expert (max,
    mean, max/mean, experts with none) and tokens per rank (max, mean)."""
    tpe = tokens_per_expert.cpu().numpy().astype(np.float64)
    tpr = tokens_per_rank.cpu().numpy().astype(np.float64)
    mean = float(tpe.mean()) if tpe.size else 0.0
    return {"pairs_per_expert_max": int(tpe.max()) if tpe.size else 0,
            "pairs_per_expert_mean": round(mean, 2),
            "expert_load_max_over_mean": round(float(tpe.max()) / mean, 3) if mean > 0 else None,
            "empty_experts": int((tpe == 0).sum()),
            "tokens_per_rank_max": int(tpr.max()) if tpr.size else 0,
            "tokens_per_rank_mean": round(float(tpr.mean()), 2) if tpr.size else 0.0}


E2E_SETS = 3  # buffer sets of the end-to-end pipeline


def measure_e2e(st: Step, spec: dict, dev, K: int, W: int, seed: int = 0) -> dict:
    """The same step through the public API with the inputs copied from pinned
    host memory every step and the combined output read back every step.

    Pipelined as a serving loop would run it: E2E_SETS buffer sets; step i's
    inputs are copied on one stream while earlier steps compute and are read
    back on another, with events ordering each buffer set's reuse (step i
    reuses the set of step i - E2E_SETS). The serial form (copy in, compute,
    copy out, one stream) is reported beside it."""
    import torch
    n = spec["num_tokens"]
    NB = E2E_SETS
    sets = [st] + [Step(spec, dev, seed) for _ in range(NB - 1)]
    # the step's inputs in pinned host memory, laid out as Step.inputs (ids,
    # weights, the row and raw scales at 256-byte-aligned offsets): one copy
    h_in = st.inputs.cpu().pin_memory()
    h_out = [torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory() for _ in range(NB)]
    h2d = h_in.numel()
    d2h = h_out[0].numel() * h_out[0].element_size()
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def copy_in(S):
        S.inputs.copy_(h_in, non_blocking=True)

    def serial(S):
        copy_in(S)
        S.run()
        h_out[0].copy_(S.out, non_blocking=True)

    def pipelined(steps, comp=comp, s_in=s_in, s_out=s_out, runs=None):
        ev_in = [torch.cuda.Event() for _ in range(NB)]
        ev_comp = [torch.cuda.Event() for _ in range(NB)]
        ev_out = [torch.cuda.Event() for _ in range(NB)]
        s_in.wait_stream(comp)
        s_out.wait_stream(comp)
        for i in range(steps):
            bset = i % NB
            S = sets[bset]
            with torch.cuda.stream(s_in):
                if i >= NB:
                    s_in.wait_event(ev_comp[bset])  # step i-NB is done with these inputs
                copy_in(S)
                ev_in[bset].record(s_in)
            comp.wait_event(ev_in[bset])
            if i >= NB:
                comp.wait_event(ev_out[bset])  # step i-NB's output has been read back
            if runs is None:
                S.run()
            else:
                for c in runs[bset]:
                    c()
            ev_comp[bset].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[bset])
                h_out[bset].copy_(S.out, non_blocking=True)
                ev_out[bset].record(s_out)
        comp.wait_stream(s_in)
        comp.wait_stream(s_out)

    # the same pipeline of G steps captured once in a CUDA graph (copies,
    # library calls and the event edges between the three streams) and
    # replayed: the host issues one launch per G steps
    G = 8 * NB
    g_comp, g_in, g_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    runs = [S.calls_on(g_comp) for S in sets]
    g_comp.wait_stream(comp)
    with torch.cuda.stream(g_comp):
        pipelined(4, g_comp, g_in, g_out, runs)
    comp.wait_stream(g_comp)
    torch.cuda.synchronize()
    graph, graph_error = torch.cuda.CUDAGraph(), None
    try:
        with torch.cuda.graph(graph, stream=g_comp):
            pipelined(G, g_comp, g_in, g_out, runs)
    except RuntimeError as err:  # reported in the line; the eager pipeline stands
        graph, graph_error = None, str(err).splitlines()[0][:200]
        torch.cuda.synchronize()
    replays = max(1, k2_graph(K, G))

    def graphed():
        for _ in range(replays):
            graph.replay()

    k2 = max(1, min(K, 200))
    res = {}
    modes = [("serial", lambda: [serial(st) for _ in range(k2)], k2),
             ("pipelined", lambda: pipelined(k2), k2)]
    if graph is not None:
        modes.append(("graph", graphed, replays * G))
    for name, fn, steps in modes:
        for _ in range(max(W, 1)):
            serial(st)
        pipelined(4)
        if graph is not None:
            graph.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(comp)
        fn()
        b.record(comp)
        torch.cuda.synchronize()
        res[name] = a.elapsed_time(b) / steps
    pipe = (f"the inputs of step i copied in while earlier steps compute and are read back "
            f"({NB} buffer sets, three streams)")
    # the faster of the two ways of issuing the same pipeline: the graph wins
    # where the host's issue rate bounds a small step, eager issue where the
    # host link does (each graph replay drains the pipeline once)
    if graph is not None and res["graph"] < res["pipelined"]:
        ms, steps = res["graph"], replays * G
        mode = f"CUDA graph of {G} pipelined steps, replayed {replays} times: {pipe}"
    else:
        ms, steps = res["pipelined"], k2
        mode = "pipelined, eager issue: " + pipe
        if graph is None:
            mode += f" (the graph capture failed: {graph_error})"
    out = {"value": round(n / (ms / 1e3), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(ms, 4), "mode": mode,
           "pipelined_eager": {"value": round(n / (res["pipelined"] / 1e3), 1),
                               "ms_per_step": round(res["pipelined"], 4), "steps": k2},
           "serial": {"value": round(n / (res["serial"] / 1e3), 1),
                      "ms_per_step": round(res["serial"], 4)}}
    if graph is not None:
        out["pipelined_graph"] = {"value": round(n / (res["graph"] / 1e3), 1),
                                  "ms_per_step": round(res["graph"], 4), "steps": replays * G}
    return out


def k2_graph(K: int, G: int) -> int:
    """Replays of a G-step graph for about min(K, 200) timed steps."""
    return -(-max(1, min(K, 200)) // G)


# ---------------------------------------------------------------- oracle arm -

def oracle_step(c: dict, spec: dict, t0: int, t1: int):
    """The oracle's layout + dispatch + combine over tokens [t0, t1)."""
    import oracle
    ids, w = c["topk_idx"][t0:t1], c["topk_weights"][t0:t1]
    e, r, h = spec["num_experts"], spec["num_ranks"], spec["hidden"]
    lay = oracle.layout(ids, e, r)
    P = lay["num_pairs"]
    if spec.get("bwd"):
        # backward with the slot map given: combine backward (expert rows are
        # zero rows here) then dispatch backward
        g = c["hidden_bf16"][t0:t1]
        y = np.zeros((max(P, 1), h), np.uint16)
        gy, _ = oracle.combine_backward(g, w, lay["slot_of"], y, max(P, 1), h)
        return oracle.dispatch_backward(gy, lay["slot_of"], h)
    if spec.get("ll"):
        # the fixed-capacity path: positions, packed payload, top-k combine
        # (the expert outputs are zero rows of the full [E * capacity] buffer)
        max_t = spec["max_tokens_per_rank"]
        ll = oracle.ll_layout(ids, e, r, max_t)
        rows = e * r * max_t
        x, s = oracle.dispatch_ll(c["hidden_bf16"][t0:t1], None, ll["ll_slot_of"], rows, oracle.BF16,
                                  oracle.FP8_E4M3_B128, h)
        y = np.zeros((rows, h), np.uint16)
        oracle.combine_topk(y, w, ll["ll_slot_of"], h)
        return x
    if spec["out_kind"] == "raw":
        rec = oracle.dispatch(ids, w, c["payload"][t0:t1], c["scales"][t0:t1], lay["slot_of"], P,
                              oracle.RAW, oracle.RAW, h, 3584, 448)
        y = np.zeros((max(P, 1), h), np.uint16)
    else:
        kind = oracle.FP8_E4M3_B128 if spec["out_kind"] == "fp8" else oracle.BF16
        rec = oracle.dispatch(ids, w, c["hidden_bf16"][t0:t1], None, lay["slot_of"], P,
                              oracle.BF16, kind, h)
        y = oracle.identity_expert(rec, spec["topk"], h, kind)
    nt = t1 - t0
    if nt % r == 0:
        oracle.combine_topk_ranks(y, ids, w, lay["slot_of"], e, r, h)
    else:
        oracle.combine_topk(y, w, lay["slot_of"], h)
    return rec


def oracle_pass_text(spec: dict) -> str:
    if spec.get("bwd"):
        return "combine backward + dispatch backward"
    if spec.get("ll"):
        return "layout + fixed-capacity layout + packed dispatch + top-k combine"
    return "layout + dispatch + combine"


# The oracle on all host cores: independent token chunks (multiples of R)
# handed to a pool of processes started with "spawn" (never forked from a
# process that holds a CUDA context). Each worker builds the seeded inputs
# once; the oracle code is the same single-threaded code.
_WORKER = {}


def _worker_init(name: str):
    spec = workload_spec(name)
    _WORKER["spec"] = spec
    _WORKER["c"] = make_inputs(spec, 0)


def _worker_chunk(bounds):
    t0, t1 = bounds
    oracle_step(_WORKER["c"], _WORKER["spec"], t0, t1)
    return t1 - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_chunks(spec: dict, tokens: int, parts: int) -> list:
    """`tokens` tokens from the workload's start cut into `parts` chunks of
    whole multiples of R tokens (wrapping around the workload when it is
    shorter)."""
    n, r = spec["num_tokens"], spec["num_ranks"]
    per = max(r, (tokens // max(parts, 1)) // r * r)
    per = min(per, n - n % r)
    out, done = [], 0
    t0 = 0
    while done < tokens:
        if t0 + per > n:
            t0 = 0
        out.append((t0, t0 + per))
        t0 += per
        done += per
    return out


class OraclePool:
    def __init__(self, spec: dict, cores: int):
        import multiprocessing as mp
        self.cores = cores
        self.pool = mp.get_context("spawn").Pool(cores, initializer=_worker_init,
                                                 initargs=(spec["name"],))
        self.pool.map(_worker_chunk, [(0, spec["num_ranks"])] * cores)  # warm every worker

    def run(self, chunks: list) -> int:
        return sum(self.pool.map(_worker_chunk, chunks, chunksize=1))

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(spec: dict, budget_s: float = 12.0) -> dict:
    """The oracle as it stands on bounded samples: single-threaded, and on all
    host cores (independent token chunks in parallel processes)."""
    c = make_inputs(spec, 0)
    n = spec["num_tokens"]
    r = spec["num_ranks"]
    t = time.perf_counter()
    oracle_step(c, spec, 0, r)
    per_tok = max((time.perf_counter() - t) / r, 1e-6)
    sample = int(min(n, max(r, budget_s / per_tok)))
    sample -= sample % r
    t = time.perf_counter()
    oracle_step(c, spec, 0, sample)
    dt = time.perf_counter() - t
    single = {"value": round(sample / dt, 2), "unit": "tokens/s", "cores": 1, "kind": "oracle",
              "sample": f"first {sample} of {n} tokens of the {spec['name']} workload, one pass of "
                        f"{oracle_pass_text(spec)} ({dt:.1f} s)"}
    cores = host_cores()
    if cores < 2:
        return single
    pool = OraclePool(spec, cores)
    try:
        tokens = int(cores * budget_s / per_tok)
        tokens = max(tokens - tokens % r, cores * r)
        chunks = oracle_chunks(spec, tokens, cores * 4)
        t = time.perf_counter()
        done = pool.run(chunks)
        dt_all = time.perf_counter() - t
    finally:
        pool.close()
    return {"value": round(done / dt_all, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} tokens of the {spec['name']} workload ({len(chunks)} chunks of "
                      f"{chunks[0][1] - chunks[0][0]} tokens, taken in order and wrapping) on "
                      f"{cores} processes, each chunk one pass of {oracle_pass_text(spec)} "
                      f"({dt_all:.1f} s)",
            "single_core": single}


def run_reference(args, spec) -> dict:
    c = make_inputs(spec, 0)
    n, r = spec["num_tokens"], spec["num_ranks"]
    K, W = args.steps, args.warmup
    t = time.perf_counter()
    oracle_step(c, spec, 0, r)
    per_tok = max((time.perf_counter() - t) / r, 1e-6)
    cores = host_cores()
    budget = args.cpu_seconds * 8  # whole reference run within a few minutes
    sample = int(min(n, max(r, cores * budget / (K + W) / per_tok)))
    sample -= sample % r
    chunks = oracle_chunks(spec, sample, cores)
    pool = OraclePool(spec, cores) if cores > 1 else None
    step = (lambda: pool.run(chunks)) if pool else (lambda: oracle_step(c, spec, 0, sample))
    try:
        for i in range(W):
            step()
        t = time.perf_counter()
        for i in range(K):
            step()
        dt = time.perf_counter() - t
    finally:
        if pool:
            pool.close()
    value = sample * K / dt
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
        "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": round(dt / K * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32 accumulate (CPU oracle)", "data": "synthetic",
        "config": {"workload": spec["text"], "num_tokens": n, "sample_tokens_per_step": sample},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"first {sample} of {n} tokens per step in {len(chunks)} chunks "
                                   f"on {cores} processes, one pass of {oracle_pass_text(spec)}"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- main -------

def whole_job(local_ms: float, local_tokens: int, world: int, device=None):
    """Whole-job time and throughput of independent replicas: the slowest
    rank's time (max over ranks) and the tokens all ranks processed divided by
    it. Collective only when world > 1 (any torch.distributed backend)."""
    total_ms = float(local_ms)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms, local_tokens * world / (total_ms / 1e3)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill",
                    choices=["prefill", "decode", "rs", "skewed", "tiny", "prefill_norm",
                             "prefill_ranks", "prefill_bwd", "decode_ll", "ag_slots",
                             "decode_sweep", "rs_sweep"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--seeds", type=int, default=5,
                    help="seeded input sets the timed steps cycle through")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="leave out the other workloads' figures from the default (prefill) line")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override N (a multiple of the workload's ranks; prefill, skewed, decode and "
                         "rs workloads), e.g. for a smaller profiling case; such a line carries no traffic")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    special = {"ag_slots": run_ag_slots, "decode_sweep": run_decode_sweep, "rs_sweep": run_rs_sweep}
    spec = workload_spec(args.workload) if args.workload not in special else None
    if args.tokens:
        if spec is None or spec["name"] in ("tiny", "decode_ll") or args.tokens % spec["num_ranks"]:
            raise SystemExit("--tokens needs a prefill, skewed, decode or rs workload and a multiple of its ranks")
        spec["num_tokens"] = args.tokens
        spec["tokens_overridden"] = True
        spec["text"] += f" (N overridden to {args.tokens})"

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if spec is None:
            raise SystemExit("the reference arm covers the dispatch/combine workloads")
        if rank == 0:
            print(json.dumps(run_reference(args, spec)), flush=True)
        return 0

    import __graft_entry__
    __graft_entry__.build()
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl")
    # No garbage-collector pass may stall the host while it enqueues timed work
    # (a stalled host leaves the GPU idle inside a step).
    gc.collect()
    gc.disable()
    try:
        line = special[args.workload](args, rank, world) if spec is None else \
            run_ours(args, spec, rank, world)
    finally:
        gc.enable()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
