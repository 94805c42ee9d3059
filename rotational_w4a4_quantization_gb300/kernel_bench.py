"""Stand-alone timing of one kernel of the library (also the target of ncu captures).

    python -m rotational_w4a4_quantization_gb300.kernel_bench --kernel gemm --workload prefill
    python -m rotational_w4a4_quantization_gb300.kernel_bench --kernel fwht --workload large
    python -m rotational_w4a4_quantization_gb300.kernel_bench --kernel fwht --n 14336   # 28 x 512
    python -m rotational_w4a4_quantization_gb300.kernel_bench --kernel kv
    python -m rotational_w4a4_quantization_gb300.kernel_bench --kernel fused --workload decode
    python -m rotational_w4a4_quantization_gb300.kernel_bench --kernel unfused --workload decode
    python -m rotational_w4a4_quantization_gb300.kernel_bench --kernel fused --workload large --rows 16
    python -m rotational_w4a4_quantization_gb300.kernel_bench --kernel attn
    python -m rotational_w4a4_quantization_gb300.kernel_bench --kernel w4a8 --workload decode
    python -m rotational_w4a4_quantization_gb300.kernel_bench --kernel w4a8 --workload prefill --group channel

Runs `--warmup` untimed launches, then `--reps` launches each timed with CUDA events on the
current stream (L2 flushed before each launch unless `--no-flush`; a GPU-side pause lets
the host enqueue ahead so the events time the kernel, not the launch), and prints the
median time with the algorithmic GB/s or TOPS.  GEMM operands are seeded random codes of
the workload's shape; rotation inputs follow the workload's outlier recipe.  `fused` times
the one-launch rotation + quantization + product of a decode batch, `unfused` the same
result from the rotation kernel followed by the GEMM kernel (two launches, one timed
region); both count the bytes of x, the packed weights and scales, and y.  `attn`
times one decode query per head over the KV workload's cache (written by the KV
kernel, 8192 tokens x 32 heads x 128) and counts the cache, the query and the output.
`w4a8` times the W4A8 product (INT8 activations, INT4 weights, one scale per group of
128, or per output channel with `--group channel`) of the workload's GEMM shape and
counts 2MNK.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

from rotational_w4a4_quantization_gb300 import build as rq_build  # noqa: E402
from rotational_w4a4_quantization_gb300 import synth  # noqa: E402


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", choices=["fwht", "kv", "gemm", "fused", "unfused", "attn", "w4a8", "w4a4g"],
                    required=True, help="w4a4g: the W4A4 product with per-group (128) weight scales, operand-form "
                                        "activations from the rotation kernel")
    ap.add_argument("--workload", choices=sorted(synth.WORKLOADS), default="prefill")
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--no-flush", action="store_true")
    ap.add_argument("--group", choices=["128", "channel"], default="128",
                    help="w4a8: weight scales per group of 128 or per output channel")
    ap.add_argument("--a-form", choices=["packed", "e4m3"], default="packed",
                    help="fwht: write the codes packed or as the product's E4M3 operand bytes; gemm: feed the "
                         "product activations in that form (made by the rotation kernel from the workload's X)")
    ap.add_argument("--rows", type=int, default=0,
                    help="gemm, fused, unfused: token rows instead of the workload's (e.g. 16 decode tokens "
                         "through the large workload's 8192 -> 28672 layer)")
    ap.add_argument("--n", type=int, default=0,
                    help="fwht: row length instead of the workload's (e.g. 14336 = 28 x 512), same rows and recipe")
    args = ap.parse_args(argv)

    rq_build.build()
    import rotational_w4a4_quantization_gb300 as rq
    rq.load_library()
    dev = torch.device("cuda")
    w = synth.WORKLOADS[args.workload]
    seed, flags = synth.SIGN_SEED, rq.RQ_SIGNS_FIRST

    if args.kernel == "fwht":
        if not w.rows:
            raise SystemExit(f"workload {w.name} has no activation")
        n = args.n or w.n
        n_out = synth._n_outliers(n) if args.n else w.n_outliers
        x = synth.activations(w.rows, n, w.x_dtype, w.data_seed, n_out, w.outlier_factor).to(dev)
        e4 = args.a_form == "e4m3"
        q = torch.empty(w.rows, n if e4 else n // 2, dtype=torch.uint8, device=dev)
        s = torch.empty((w.rows, 2) if e4 else (w.rows,), dtype=torch.float32, device=dev)   # e4m3: scale, code sum
        fl = flags | (rq.RQ_E4M3_CODES if e4 else 0)
        fn = lambda: rq.fwht_quant(x, seed, fl, q=q, scales=s)
        work, unit = w.rows * (n * x.element_size() + (n if e4 else n // 2) + (8 if e4 else 4)), "GB/s"
        what = f"fwht_quant {w.rows}x{n} {str(x.dtype).split('.')[-1]}{' e4m3 codes' if e4 else ''}"
    elif args.kernel == "kv":
        kw = synth.KV
        k, v = synth.kv_pair(kw.kv_tokens, kw.kv_heads, kw.kv_head_dim, kw.data_seed,
                             kw.kv_outliers_per_head, kw.kv_outlier_factor)
        k, v = k.to(dev), v.to(dev)
        out = rq.kv_rotate_quant(k, v, seed, flags)
        fn = lambda: rq.kv_rotate_quant(k, v, seed, flags, out=out)
        T, H, D = k.shape
        work, unit = 2 * T * H * (D * 2 + D // 2 + 4), "GB/s"
        what = f"kv_rotate_quant {T}x{H}x{D} bf16"
    elif args.kernel == "w4a8":
        if not w.gemm_n:
            raise SystemExit(f"workload {w.name} has no GEMM")
        M, K, N = w.rows, w.n, w.gemm_n
        g8 = torch.Generator().manual_seed(1000 + w.data_seed)
        a8 = torch.randint(-128, 128, (M, K), dtype=torch.int8, generator=g8).to(dev)
        s8 = (torch.rand(M, generator=g8) + 0.05).to(dev)
        wq, _ = synth.random_codes(N, K, 1001 + w.data_seed)
        per_channel = args.group == "channel"
        sg = (torch.rand(N, generator=g8) if per_channel else torch.rand(N, K // 128, generator=g8)) + 0.05
        sg, wq = sg.to(dev), wq.to(dev)
        y = torch.empty(M, N, dtype=torch.float16, device=dev)
        fn = lambda: rq.w4a8_gemm(a8, s8, wq, sg, out=y)
        work, unit = 2 * M * N * K, "TOPS"
        what = f"w4a8_gemm {M}x{K}x{N} {'per-channel' if per_channel else 'per-group-128'} fp16"
    elif args.kernel == "w4a4g":
        if not w.gemm_n:
            raise SystemExit(f"workload {w.name} has no GEMM")
        M, K, N = w.rows, w.n, w.gemm_n
        x = synth.activations(M, K, w.x_dtype, w.data_seed, w.n_outliers, w.outlier_factor).to(dev)
        ae, sa2 = rq.fwht_quant(x, seed, flags | rq.RQ_E4M3_CODES)
        wq, _ = synth.random_codes(N, K, 1001 + w.data_seed)
        g8 = torch.Generator().manual_seed(1002 + w.data_seed)
        sg = (torch.rand(N, K // 128, generator=g8) + 0.05).to(dev)
        wq = wq.to(dev)
        y = torch.empty(M, N, dtype=torch.float16, device=dev)
        fn = lambda: rq.w4a4_gemm(ae, sa2, wq, sg, out=y)
        work, unit = 2 * M * N * K, "TOPS"
        what = f"w4a4_gemm {M}x{K}x{N} per-group-128 fp16 (e4m3 activations)"
    elif args.kernel == "attn":
        kw = synth.KV
        k, v = synth.kv_pair(kw.kv_tokens, kw.kv_heads, kw.kv_head_dim, kw.data_seed,
                             kw.kv_outliers_per_head, kw.kv_outlier_factor)
        cache = rq.kv_rotate_quant(k.to(dev), v.to(dev), seed, flags)
        T, H, D = k.shape
        qd = synth.kv_pair(1, H, D, kw.data_seed + 500, kw.kv_outliers_per_head, kw.kv_outlier_factor)[0].to(dev)
        o = torch.empty(1, H, D, dtype=torch.float32, device=dev)
        fn = lambda: rq.attn_decode(qd, cache, seed, flags, out=o)
        work, unit = 2 * T * H * (D // 2 + 4) + H * D * 2 + H * D * 4, "GB/s"
        what = f"attn_decode 1 query x {H} heads x {D} over {T} cached tokens"
    elif args.kernel in ("fused", "unfused"):
        if not w.gemm_n or not w.rows:
            raise SystemExit(f"workload {w.name} has no activation GEMM")
        M, K, N = args.rows or w.rows, w.n, w.gemm_n
        x = synth.activations(M, K, w.x_dtype, w.data_seed, w.n_outliers, w.outlier_factor).to(dev)
        wq, sw = synth.random_codes(N, K, 1001 + w.data_seed)
        wq, sw = wq.to(dev), sw.to(dev)
        y = torch.empty(M, N, dtype=torch.float16, device=dev)
        if args.kernel == "fused":
            fn = lambda: rq.fwht_quant_gemm(x, seed, flags, wq, sw, out=y)
        else:
            q = torch.empty(M, K // 2, dtype=torch.uint8, device=dev)
            s = torch.empty(M, dtype=torch.float32, device=dev)

            def fn():
                rq.fwht_quant(x, seed, flags, q=q, scales=s)
                rq.w4a4_gemm(q, s, wq, sw, out=y)
        work, unit = M * K * x.element_size() + N * K // 2 + 4 * N + 2 * M * N, "GB/s"
        what = f"{args.kernel} rotate+quant+gemm {M}x{K}x{N} {str(x.dtype).split('.')[-1]} -> fp16"
    else:
        if not w.gemm_n:
            raise SystemExit(f"workload {w.name} has no GEMM")
        M, K, N = args.rows or w.rows, w.n, w.gemm_n
        aq, sa = synth.random_codes(M, K, 1000 + w.data_seed)
        wq, sw = synth.random_codes(N, K, 1001 + w.data_seed)
        d = [t.to(dev) for t in (aq, sa, wq, sw)]
        if args.a_form == "e4m3":
            x = synth.activations(M, K, w.x_dtype, w.data_seed, w.n_outliers, w.outlier_factor).to(dev)
            d[0], d[1] = rq.fwht_quant(x, seed, flags | rq.RQ_E4M3_CODES)
        y = torch.empty(M, N, dtype=torch.float16, device=dev)
        fn = lambda: rq.w4a4_gemm(*d, out=y)
        work, unit = 2 * M * N * K, "TOPS"
        what = f"w4a4_gemm {M}x{K}x{N} fp16{' (e4m3 activations)' if args.a_form == 'e4m3' else ''}"

    flush = torch.empty(2 * torch.cuda.get_device_properties(dev).L2_cache_size, dtype=torch.uint8,
                        device=dev)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    ev = []
    for i in range(args.reps):
        if not args.no_flush:
            flush.fill_(i & 0xFF)
        torch.cuda._sleep(400_000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    assert rq.sync_status() == 0
    times = sorted(a.elapsed_time(b) * 1e-3 for a, b in ev)
    med = times[len(times) // 2]
    rate = work / med / (1e9 if unit == "GB/s" else 1e12)
    mean = sum(times) / len(times)   # events tick in ~2 us steps here: the mean of many reps resolves finer
    print(f"{what}: median {med * 1e6:.1f} us  mean {mean * 1e6:.2f} us  min {times[0] * 1e6:.1f} us  "
          f"{rate:.1f} {unit} (median)")


if __name__ == "__main__":
    main()
