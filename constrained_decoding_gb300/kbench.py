"""Kernel-level timing of the projection GEMMs through the C ABI
(`pcd_k_gemm`, `pcd_k_gemm_swap`): the shapes of the decoder's projections,
timed over back-to-back launches on one stream (as a pass issues them), with
rotating weight copies so every launch streams its weights from HBM.

    python -m constrained_decoding_gb300.kbench [--cases NAME ...]

Prints one JSON line per (shape, kernel form): microseconds per launch,
weight-streaming GB/s and TFLOP/s.  Needs a GPU and the built library.
"""
from __future__ import annotations

import argparse
import json

# name: (M, N, K, epilogue, forms); epilogue 1 f32 add, 2 f32 atomic, 3 SwiGLU.
# Forms: ("tile", mt, bn, splits) row tiles (mt 0 = the library's choice,
# mt 3 = CTA pairs), ("swap", splits) weight-streaming form.
CASES = {
    "gate_up_313": (313, 17920, 1536, 3, [("tile", 0, 0, 1), ("tile", 2, 256, 1), ("tile", 3, 256, 1), ("swap", 1)]),
    "down_313": (313, 1536, 8960, 2, [("tile", 1, 256, 8), ("tile", 2, 256, 8), ("swap", 0)]),
    "gate_up_512": (512, 17920, 1536, 3, [("tile", 0, 0, 1), ("tile", 3, 256, 1), ("swap", 1)]),
    "gate_up_825": (825, 17920, 1536, 3, [("tile", 0, 0, 1), ("tile", 2, 256, 1), ("tile", 3, 256, 1)]),
    "down_825": (825, 1536, 8960, 2, [("tile", 1, 256, 3), ("tile", 3, 256, 3)]),
    "gate_up_8192": (8192, 17920, 1536, 3, [("tile", 0, 0, 1), ("tile", 3, 256, 1)]),
    "down_8192": (8192, 1536, 8960, 2, [("tile", 1, 256, 1), ("tile", 3, 256, 1)]),
    "qkv_8192": (8192, 2048, 1536, 1, [("tile", 0, 0, 1), ("tile", 1, 128, 1)]),
    "readout_117": (117, 151936, 1536, 3, [("tile", 0, 0, 1)]),
}


def time_launches(fn, n=20, reps=5):
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    ts = []
    for _ in range(reps):
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e3 / n)
    ts.sort()
    return ts[len(ts) // 2]


def run_case(lib, name, M, N, K, epi, forms, n_copies):
    import torch
    s = torch.cuda.current_stream().cuda_stream
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(0)
    a = (torch.randn(M, K, device="cuda", generator=g) * 0.5).half()
    ws = [(torch.randn(N, K, device="cuda", generator=g) * 0.05).half() for _ in range(n_copies)]
    out = torch.zeros(M, N // 2 if epi == 3 else N, dtype=torch.float16 if epi == 3 else torch.float32,
                      device="cuda")
    for form in forms:
        k = {"i": 0}

        def launch():
            w = ws[k["i"] % n_copies]
            k["i"] += 1
            if form[0] == "tile":
                rc = lib.pcd_k_gemm(a.data_ptr(), M, K, w.data_ptr(), N, K, K, epi, out.data_ptr(), out.shape[1],
                                    form[1], form[2], form[3], err.data_ptr(), s)
            else:
                rc = lib.pcd_k_gemm_swap(a.data_ptr(), None, M, K, w.data_ptr(), N, K, K, epi, out.data_ptr(),
                                         out.shape[1], form[1], err.data_ptr(), s)
            if rc != 0:
                raise RuntimeError(f"{name} {form}: status {rc}")

        us = time_launches(launch)
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise RuntimeError(f"{name} {form}: device error {int(err.item())}")
        print(json.dumps({"case": name, "M": M, "N": N, "K": K, "form": list(form), "us_per_launch": round(us, 2),
                          "weight_gbs": round(N * K * 2 / us / 1e3, 1),
                          "tflops": round(2.0 * M * N * K / us / 1e6, 1)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--cases", nargs="*", default=list(CASES))
    args = ap.parse_args()
    from constrained_decoding_gb300 import load
    lib = load()
    for name in args.cases:
        M, N, K, epi, forms = CASES[name]
        # enough weight copies that a launch never finds its weights in the 126 MB L2
        n_copies = max(2, min(4, -(-256 * 2**20 // (N * K * 2))))
        run_case(lib, name, M, N, K, epi, forms, n_copies)


if __name__ == "__main__":
    main()
