"""Decode-step driver: the 197 projection GEMVs of one Qwen2.5-1.5B-shaped decode step, run back
to back on one stream and replayed as one CUDA graph ("Do Quantization and Sparsity make LLM
Inference Faster ?", section "What we did": eight shapes, 197 GEMVs per token; "My Triton Kernel
Ties bitsandbytes", section "What's next": CUDA graphs around the decode step).

Weights are synthetic (synth.weights, N(0, 0.02)) and quantised on the GPU by libw4.  All
activations live in one contiguous device arena and all outputs in another, so a host round trip
is one copy each way.  Each GEMV reads x only after every earlier GEMV of the step has completed
(stream order + programmatic dependent launch), as in a real decode step.
"""
from __future__ import annotations

import numpy as np

from . import synth
from . import _lib
import weight_only_bit_gb300 as w4


def _align8(n: int) -> int:
    return (n + 7) // 8 * 8


class DecodeStep:
    def __init__(self, fmt: str = "nf4", batch: int = 1, device: str = "cuda:0", blocksize: int | None = None,
                 outlier_frac: float = 0.0, layers: int = synth.N_LAYERS, lm_head: bool = True,
                 levels: str = "grouped"):
        """levels="grouped": GEMVs reading the same activation form one level (q,k,v / o / gate,up /
        down / lm_head: 113 levels for the full step); levels="strict": every GEMV waits for the one
        before it (197 levels)."""
        import torch
        self.torch = torch
        self.fmt = fmt
        self.format = {"nf4": _lib.W4_FMT_NF4, "int4": _lib.W4_FMT_INT4, "fp4": _lib.W4_FMT_FP4}[fmt]
        self.bs = blocksize or {"nf4": 64, "int4": 128, "fp4": 32}[fmt]
        self.M = batch
        self.dev = torch.device(device)
        self.outlier_frac = outlier_frac
        self.gemvs = [g for g in synth.decode_step_gemvs()
                      if (g[1] != "lm_head" and g[0] < layers) or (g[1] == "lm_head" and lm_head)]
        # x slots: (layer, slot) -> offset in the x arena
        self.x_off = {}
        off = 0
        for layer, proj, n, k in self.gemvs:
            key = (layer, synth.X_SLOT[proj])
            if key not in self.x_off:
                self.x_off[key] = (off, k)
                off += _align8(batch * k)
        self.x_elems = off
        self.y_off = []
        off = 0
        for layer, proj, n, k in self.gemvs:
            self.y_off.append(off)
            off += _align8(batch * n)
        self.y_elems = off
        self.levels = []
        lev, prev = -1, None
        for i, (layer, proj, n, k) in enumerate(self.gemvs):
            key = (layer, synth.X_SLOT[proj])
            if levels == "strict" or key != prev:
                lev += 1
            prev = key
            self.levels.append(lev)
        self.code = None
        self.packed, self.scales = [], []
        self.step = None

    # ------------------------------------------------------------------ setup
    def build(self, seed_offset: int = 0):
        torch = self.torch
        if self.format == _lib.W4_FMT_NF4:
            st, c = w4.w4_nf4_codebook()
            w4.check(st, "codebook")
            self.code = torch.tensor(c, dtype=torch.float32, device=self.dev)
        self.x = torch.empty(self.x_elems, dtype=torch.float16, device=self.dev)
        self.y = torch.zeros(self.y_elems, dtype=torch.float16, device=self.dev)
        xs = np.zeros(self.x_elems, dtype=np.float16)
        for (layer, slot), (o, k) in self.x_off.items():
            xs[o:o + self.M * k] = synth.activations(synth.x_seed(layer, slot, self.M), self.M, k).ravel()
        self.x.copy_(torch.from_numpy(xs))
        self.x_host = xs
        for layer, proj, n, k in self.gemvs:
            w = synth.weights(synth.weight_seed(layer, proj) + seed_offset, n, k, outlier_frac=self.outlier_frac)
            W = torch.from_numpy(w).to(self.dev)
            packed = torch.empty((n, k // 2), dtype=torch.uint8, device=self.dev)
            if self.format == _lib.W4_FMT_NF4:
                sc = torch.empty((n, k // self.bs), dtype=torch.float32, device=self.dev)
                w4.check(w4.w4_quantize_nf4(W, packed, sc, self.code, n, k, self.bs), f"quantize {proj}")
            else:
                sc = torch.empty((n, k // self.bs), dtype=torch.float16, device=self.dev)
                quant = w4.w4_quantize_int4 if self.format == _lib.W4_FMT_INT4 else w4.w4_quantize_fp4
                w4.check(quant(W, packed, sc, n, k, self.bs), f"quantize {proj}")
            self.packed.append(packed)
            self.scales.append(sc)
            del W
        torch.cuda.synchronize(self.dev)
        return self

    def descriptors(self):
        d = []
        for i, (layer, proj, n, k) in enumerate(self.gemvs):
            xo, _ = self.x_off[(layer, synth.X_SLOT[proj])]
            d.append(dict(format=self.format, packed=self.packed[i], scales=self.scales[i], codebook=self.code,
                          x=self.x.data_ptr() + 2 * xo, y=self.y.data_ptr() + 2 * self.y_off[i],
                          M=self.M, N=n, K=k, blocksize=self.bs, level=self.levels[i]))
        return d

    def capture(self):
        torch = self.torch
        nbytes = w4.w4_step_workspace_bytes(len(self.gemvs))
        self.workspace = torch.zeros(nbytes // 4, dtype=torch.int32, device=self.dev)
        st, h = w4.w4_step_create(self.descriptors(), self.workspace)
        w4.check(st, "step create")
        self.step = h
        return self

    def counters(self):
        """The level counters at the start of the step workspace (one per GEMV, plus one)."""
        return self.workspace[: len(self.gemvs) + 1]

    def launch(self, stream=None):
        return w4.w4_step_launch(self.step, stream)

    def run_host(self, x_host, y_host, stream=None):
        """One step from and to host buffers (pinned tensors of the x and y arenas' sizes) through
        the library's w4_step_run_host."""
        return w4.w4_step_run_host(self.step, x_host, self.x, self.x_elems * 2, y_host, self.y, self.y_elems * 2,
                                   stream)

    def enqueue_eager(self, stream=None):
        """One launch per GEMV, back to back (the same results, without the persistent step)."""
        return w4.w4_gemv_sequence(self.descriptors(), stream)

    def close(self):
        if self.step is not None:
            w4.w4_step_destroy(self.step)
            self.step = None

    # ------------------------------------------------------------------ accounting
    def scale_bytes(self, n: int, k: int) -> int:
        return n * (k // self.bs) * (4 if self.format == _lib.W4_FMT_NF4 else 2)

    def gemv_bytes(self, i: int) -> int:
        """Algorithmic bytes of GEMV i: packed weights + scales + x + y (each touched once)."""
        _, _, n, k = self.gemvs[i]
        return n * k // 2 + self.scale_bytes(n, k) + 2 * self.M * k + 2 * self.M * n

    def bytes_per_step(self) -> int:
        return sum(self.gemv_bytes(i) for i in range(len(self.gemvs)))

    def y_of(self, i: int):
        _, _, n, _ = self.gemvs[i]
        o = self.y_off[i]
        return self.y[o:o + self.M * n].view(self.M, n)

    def x_of(self, i: int):
        layer, proj, n, k = self.gemvs[i]
        o, _ = self.x_off[(layer, synth.X_SLOT[proj])]
        return self.x_host[o:o + self.M * k].reshape(self.M, k)


def _main():
    """Run a decode step on cuda:0 and print its device time (also the workload the ncu
    summaries under profiles/ were captured on)."""
    import argparse
    import torch
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--fmt", default="nf4", choices=["nf4", "int4", "fp4"])
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--layers", type=int, default=synth.N_LAYERS)
    ap.add_argument("--no-lm-head", action="store_true")
    ap.add_argument("--levels", default="grouped", choices=["grouped", "strict"])
    ap.add_argument("--launch-per-gemv", action="store_true", help="one launch per GEMV instead of one per step")
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    a = ap.parse_args()
    from weight_only_bit_gb300 import build as _b
    _b.build()
    st = DecodeStep(a.fmt, a.batch, "cuda:0", layers=a.layers, lm_head=not a.no_lm_head, levels=a.levels).build()
    stream = torch.cuda.Stream()
    if a.launch_per_gemv:
        run = lambda: w4.check(st.enqueue_eager(stream))
    else:
        st.capture()
        run = lambda: w4.check(st.launch(stream))
    for _ in range(a.warmup):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(a.steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    w4.check(w4.w4_device_check(stream))
    ms = e0.elapsed_time(e1) / a.steps
    print(f"{a.fmt} batch {a.batch}, {len(st.gemvs)} GEMVs, {st.levels[-1] + 1} levels: {ms * 1e3:.1f} us/step, "
          f"{st.bytes_per_step() / (ms * 1e-3) / 1e9:.1f} GB/s")
    st.close()


if __name__ == "__main__":
    _main()
