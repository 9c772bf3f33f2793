"""Run one operation of the library on a named synthetic workload, a few times.

A small driver for profilers and quick timing: it allocates only what the
chosen operation needs, runs it ``--iters`` times on cuda:0 and prints the
mean CUDA-event time of the launches after the first.

  python -m exact_tiled_attention_attn_gb300.run_op --op prefill --workload gqa-llama --iters 3
  python -m exact_tiled_attention_attn_gb300.run_op --op backward --iters 3
  python -m exact_tiled_attention_attn_gb300.run_op --op decode --iters 3
  python -m exact_tiled_attention_attn_gb300.run_op --op decode_fp8 --iters 3
  python -m exact_tiled_attention_attn_gb300.run_op --op rmsnorm --iters 3
  python -m exact_tiled_attention_attn_gb300.run_op --op rmsnorm_residual --iters 3
  python -m exact_tiled_attention_attn_gb300.run_op --op kv_quant --iters 3

Workloads (seeded N(0,1) bf16 inputs):
  single-head  causal 1 x 1 x 256 x 64
  mha-gpt2     non-causal B8 H12 T4096 d64
  gqa-qwen     causal B1 Hq16 Hkv8 T4096 d128
  gqa-llama    causal B2 Hq32 Hkv8 T8192 d128 (default for prefill)
  decode-llama B16 Hq32 Hkv8 d128, lengths ~U[8192, 32768] (decode)
  norm-qwen    X[4096, 1024] (rmsnorm, rmsnorm_residual)
  kv_quant quantises the K cache of decode-llama to E4M3 (one scale per (sequence, head))
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PREFILL_WORKLOADS = {"single-head": "SINGLE_HEAD", "mha-gpt2": "MHA_GPT2", "gqa-qwen": "GQA_QWEN",
                     "gqa-llama": "GQA_LLAMA"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["prefill", "backward", "decode", "decode_fp8", "rmsnorm", "rmsnorm_residual",
                                           "kv_quant"], required=True)
    ap.add_argument("--workload", default=None)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--splits", type=int, default=None,
                    help="decode: split count; 0 = the balanced schedule (default: the library default count)")
    ap.add_argument("--rows", type=int, default=0, help="rmsnorm: rows T of X[T, 1024] (default: the workload's)")
    args = ap.parse_args(argv)

    import torch
    import workloads as W
    import exact_tiled_attention_attn_gb300 as attn
    from exact_tiled_attention_attn_gb300.build import build

    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.op == "prefill":
        shp = getattr(W, PREFILL_WORKLOADS[args.workload or "gqa-llama"])
        q, k, v = W.attention_inputs(shp)[:3]
        q, k, v = q.to(dev), k.to(dev), v.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)

        def run():
            attn.fwd(q, k, v, causal=shp.causal, scale=shp.scale, out=o, lse=lse)
        work, unit = shp.flops() / 1e12, "TFLOP/s"
    elif args.op == "backward":
        shp = getattr(W, PREFILL_WORKLOADS[args.workload or "gqa-llama"])
        q, k, v = W.attention_inputs(shp)[:3]
        q, k, v = q.to(dev), k.to(dev), v.to(dev)
        do = W.grad_output(shp.B, shp.Hq, shp.T, shp.d, shp.seed).to(dev)
        o, lse = attn.fwd(q, k, v, causal=shp.causal, scale=shp.scale)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

        def run():
            attn.bwd(q, k, v, o, lse, do, causal=shp.causal, scale=shp.scale, dq=dq, dk=dk, dv=dv)
        work, unit = 2.5 * shp.flops() / 1e12, "TFLOP/s (5-GEMM algorithmic)"
    elif args.op in ("decode", "decode_fp8"):
        shp = W.DECODE_LLAMA
        q, kc, vc, sl = W.decode_inputs(shp)
        q, kc, vc, sld = q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev)
        S = args.splits if args.splits is not None else attn.default_splits(shp.B, shp.Hkv, shp.Lcap)
        ws = torch.empty(attn.decode_workspace_size(shp.B, shp.Hq, shp.d, S), dtype=torch.uint8, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty(shp.B, shp.Hq, dtype=torch.float32, device=dev)
        if args.op == "decode":
            def run():
                attn.decode(q, kc, vc, sld, scale=shp.scale, num_splits=S, workspace=ws, out=o, lse=lse)
            work, unit = 4 * shp.Hkv * shp.d * int(sl.sum()) / 1e9, "GB/s (KV stream)"
        else:  # the cache quantised to E4M3 once, outside the timed launches
            kq, ks = attn.kv_quantize_fp8(kc)
            vq, vs = attn.kv_quantize_fp8(vc)
            del kc, vc

            def run():
                attn.decode_fp8(q, kq, vq, ks, vs, sld, scale=shp.scale, num_splits=S, workspace=ws, out=o, lse=lse)
            work, unit = 2 * shp.Hkv * shp.d * int(sl.sum()) / 1e9, "GB/s (E4M3 KV stream)"
    elif args.op == "kv_quant":
        shp = W.DECODE_LLAMA
        kc = W.decode_inputs(shp)[1].to(dev)
        codes = torch.empty(kc.shape, dtype=torch.uint8, device=dev)
        sc = torch.empty(shp.B, shp.Hkv, dtype=torch.float32, device=dev)

        def run():
            attn.kv_quantize_fp8(kc, codes=codes, scale=sc)
        # the whole bf16 cache is read twice (amax pass, encode pass) and the codes written once
        work, unit = (2 * kc.numel() * 2 + kc.numel()) / 1e9, "GB/s (2 reads of the bf16 cache + codes)"
    else:
        shp = W.NORM_QWEN
        if args.rows > 0:
            shp = W.NormShape(f"RMSNorm X[{args.rows},{shp.D}]", args.rows, shp.D, shp.eps, shp.seed)
        x, w = W.norm_inputs(shp)
        x, w = x.to(dev), w.to(dev)
        y = torch.empty_like(x)
        if args.op == "rmsnorm":
            def run():
                attn.rmsnorm(x, w, eps=shp.eps, out=y)
            work, unit = shp.hbm_bytes() / 1e9, "GB/s"
        else:
            r = torch.flip(x, dims=[0]).contiguous()
            h = torch.empty_like(x)

            def run():
                attn.rmsnorm_residual(x, r, w, eps=shp.eps, out=y, h=h)
            work, unit = (8 * shp.T * shp.D + 2 * shp.D) / 1e9, "GB/s"

    run()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    n = max(1, args.iters - 1)
    ev[0].record()
    for _ in range(n):
        run()
    ev[1].record()
    torch.cuda.synchronize()
    status = attn.last_device_error()
    ms = ev[0].elapsed_time(ev[1]) / n
    print(f"{args.op} {shp.name}: {ms:.4f} ms/launch, {work / (ms * 1e-3):.1f} {unit}, device status {status}")
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
