"""Run one kernel of the path on a small case, for ncu captures.

  python -m quantized_weight_matvec_gb300.profile_case --kernel f8 --rows 65536 --iters 3

Kernels: f8 (E4M3 head-shaped rows x 4096, scales [rows/128, 32]), i8
(int8 rows x 4096, per-16 E8M0 group scales), cq2
(2-bit rows x 512, group 128, the table kernel), cqvec (--bits-bit rows x
512, group 64, the vectorised kernel), gather (64 rows of a 32768 x 512
2-bit matrix), prepare, topk (top-64 temperature sampling over --rows
normal logits per vector).  Inputs are seeded synthetic data; the case is chosen
larger than L2 but a few hundred MB at most.  Prints one checksum line and
no timings: numbers taken under a profiler are not measurements.
"""
from __future__ import annotations

import argparse

import torch

from . import qmv, synth


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", choices=["f8", "i8", "cq2", "cqvec", "gather", "prepare", "topk"], required=True)
    ap.add_argument("--bits", type=int, default=4)
    ap.add_argument("--rows", type=int, default=65536)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args(argv)
    qmv.load()
    dev = torch.device("cuda", 0)
    if args.kernel == "f8":
        f = synth.f8_inputs(5, args.rows, 4096, max(1, args.rows // 128), 32, 118, 132,
                            batch=args.batch)
        w, s, x = (torch.from_numpy(a).to(dev) for a in (f.w, f.scale, f.x))
        y = torch.empty((args.batch, args.rows), device=dev)
        for _ in range(args.iters):
            qmv.f8_matvec_t(w, s, x, out=y)
        out = y
    elif args.kernel == "i8":
        f = synth.i8_inputs(7, args.rows, 4096, 110, 124, batch=args.batch)
        w, s, x = (torch.from_numpy(a).to(dev) for a in (f.w, f.scale, f.x))
        y = torch.empty((args.batch, args.rows), device=dev)
        for _ in range(args.iters):
            qmv.i8_matvec_t(w, s, x, out=y)
        out = y
    elif args.kernel == "topk":
        g = torch.Generator(device="cpu").manual_seed(0)
        y = (torch.randn((args.batch, args.rows), generator=g) * 3).to(dev)
        u = torch.rand(args.batch, generator=g).to(dev)
        for _ in range(args.iters):
            idx, val, prob, tok = qmv.topk_sample_t(y, 64, 1.0, u)
        out = prob
    elif args.kernel == "cqvec":
        c = synth.cq_inputs(2, args.rows, 512, 64, args.bits, batch=args.batch)
        m = qmv.CQMatrix.from_numpy(c, device=dev)
        p = qmv.cq_prepare_t(m, torch.from_numpy(c.x).to(dev))
        for _ in range(args.iters):
            out = qmv.cq_matvec_t(m, p)
    else:
        rows = args.rows if args.kernel == "cq2" else 32768
        c = synth.cq_inputs(3, rows, 500, 128, 2, batch=args.batch, x_scale=3.0, gather=64)
        m = qmv.CQMatrix.from_numpy(c, device=dev)
        x = torch.from_numpy(c.x).to(dev)
        p = qmv.cq_prepare_t(m, x)
        for _ in range(args.iters):
            if args.kernel == "cq2":
                out = qmv.cq_matvec_t(m, p)
            elif args.kernel == "gather":
                out = qmv.cq_dequantize_row_t(m, torch.from_numpy(c.rows).to(dev))
            else:
                out = qmv.cq_prepare_t(m, x, out=p)
    torch.cuda.synchronize()
    print("checksum %.6e" % float(out.double().abs().sum()))


if __name__ == "__main__":
    main()
