"""L1-regularised training of one sparse FFN block on synthetic data.

"Sparser, Faster, Lighter Transformer Language Models", Resumo Técnico §2,
"Técnicas de Treinamento": a plain L1 penalty on the ReLU activations of the
feed-forward layers drives their sparsity up during training. This demo shows
that on one layer, teacher-student style, with the library doing the layer's
work:

  target  y* = teacher(x): a narrow dense ReLU FFN (64 hidden units), computed
          with twell_dense_ffn_fwd on the tensor cores;
  student y  = relu(x W_up^T + b) W_down with d_ff hidden units, forward with
          twell_ffn_fwd (TwELL packed in the up-projection's epilogue);
  loss    L = 1/(2M) sum ||y - y*||^2 + lam/M * sum |h|;
  grads   twell_ffn_bwd with dy = (y - y*)/M and l1 = lam/M;
  update  Adam on fp32 master weights (torch; the optimiser is not part of the
          library), rounded to bf16 for the next step.

Each step draws a fresh batch x ~ N(0, 1) on the GPU. The printed table shows
the loss falling while the hidden density falls with it, and the step time
following the density. Run with ``python -m
activation_sparse_transformer_tcgen05_gb300.train_demo [--steps N] [--lam L]``.
"""
from __future__ import annotations

import argparse
import time

import torch

from . import twell as tw


def _bits(t: torch.Tensor) -> torch.Tensor:
    """bf16 bit pattern (int16 view) of an fp32 tensor, rounded to nearest even."""
    return t.to(torch.bfloat16).view(torch.int16).contiguous()


def train(steps: int = 1000, M: int = 4096, d: int = 1024, F: int = 4096, T: int = 128, lam: float = 0.05,
          lr: float = 2e-3, teacher_units: int = 64, seed: int = 0, log_every: int = 100, verbose: bool = True):
    """Runs the demo; returns the per-step history (loss, density, ms)."""
    dev = "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    Ft = teacher_units
    Tu = torch.randn(Ft, d, device=dev, generator=g) / d ** 0.5
    Td = torch.randn(Ft, d, device=dev, generator=g) / Ft ** 0.5
    teacher = (_bits(Tu), torch.zeros(Ft, device=dev), _bits(Td))
    params = [torch.randn(F, d, device=dev, generator=g) / d ** 0.5,  # W_up
              torch.zeros(F, device=dev),                              # b
              torch.randn(F, d, device=dev, generator=g) / F ** 0.5]  # W_down
    m = [torch.zeros_like(p) for p in params]
    v = [torch.zeros_like(p) for p in params]
    b1, b2, eps = 0.9, 0.999, 1e-8

    buf = tw.TwellBuffers(M, F, T, M * F)
    ws_f = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_FWD, M, d, F, T, M * F), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(tw.twell_workspace_bytes(tw.OP_FFN_BWD, M, d, F, T, M * F), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    y = torch.empty(M, d, dtype=torch.int16, device=dev)
    ys = torch.empty(M, d, dtype=torch.int16, device=dev)
    ht = torch.empty(M, Ft, dtype=torch.int16, device=dev)
    dx = torch.empty(M, d, dtype=torch.int16, device=dev)
    dWu = torch.empty(F, d, dtype=torch.float32, device=dev)
    dWd = torch.empty(F, d, dtype=torch.float32, device=dev)
    db = torch.empty(F, dtype=torch.float32, device=dev)

    hist = []
    if verbose:
        print(f"{'step':>6} {'loss':>10} {'density':>9} {'ms/step':>8}")
    for s in range(1, steps + 1):
        x = _bits(torch.randn(M, d, device=dev, generator=g))
        Wu, b, Wd = _bits(params[0]), params[1].contiguous(), _bits(params[2])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tw.twell_dense_ffn_fwd(x, teacher[0], teacher[1], teacher[2], ht, ys, st)
        e0.record()
        tw.twell_ffn_fwd(x, Wu, None, b, Wd, T, buf, y, ws_f, st)
        r = y.view(torch.bfloat16).float() - ys.view(torch.bfloat16).float()
        dy = _bits(r / M)
        tw.twell_ffn_bwd(x, Wu, Wd, buf, dy, lam / M, dx, dWu, dWd, db, ws_b, st)
        e1.record()
        for i, grad in enumerate((dWu, db, dWd)):
            m[i].mul_(b1).add_(grad, alpha=1 - b1)
            v[i].mul_(b2).addcmul_(grad, grad, value=1 - b2)
            step = lr / (1 - b1 ** s)
            params[i].addcdiv_(m[i], (v[i] / (1 - b2 ** s)).sqrt_().add_(eps), value=-step)
        if s % log_every == 0 or s == 1 or s == steps:
            code = tw.twell_check(st)
            if code != 0:
                raise RuntimeError(f"device status {code}: {tw.twell_status_string(code)}")
            loss = 0.5 * float((r * r).sum()) / M
            density = float(buf.nnz.sum()) / (M * F)
            ms = e0.elapsed_time(e1)
            hist.append({"step": s, "loss": loss, "density": density, "ms": ms})
            if verbose:
                print(f"{s:6d} {loss:10.4f} {density:9.4f} {ms:8.3f}")
    return hist


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--lam", type=float, default=0.05)
    ap.add_argument("--lr", type=float, default=2e-3)
    ap.add_argument("--M", type=int, default=4096)
    ap.add_argument("--d", type=int, default=1024)
    ap.add_argument("--F", type=int, default=4096)
    args = ap.parse_args(argv)
    t0 = time.time()
    train(args.steps, args.M, args.d, args.F, lam=args.lam, lr=args.lr)
    print(f"wall {time.time() - t0:.1f} s")


if __name__ == "__main__":
    main()
