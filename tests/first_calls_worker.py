"""Makes the library's first calls in this process from several host threads
at once: each thread runs a product on a different kernel variant (so each
kernel's one-time shared-memory set-up, the pair kernels' occupancy queries
and the device's cached properties are first reached concurrently), then all
results are compared with the oracle.

    python first_calls_worker.py

Exit status 0 when every product is within its bound (run by
test_first_calls_threads.py in a fresh process)."""
import os
import sys
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
sys.path.insert(0, ROOT)
sys.path.insert(0, HERE)

import torch  # noqa: E402

import dense_gemm_14_gb300 as g14  # noqa: E402
import oracle  # noqa: E402
from dense_gemm_14_gb300 import inputs  # noqa: E402

TOL = {"f32": 1e-5, "bf16": 4e-3, "f16": 4e-3}
# (dtype, M, N, K, entry): the fp32 large and small-tile kernels, the one-SM
# tensor kernel with 64- and 128-row tiles, the pair kernel, the TF32 kernels
CASES = [("f32", 2048, 2048, 64, "gemm_f32"), ("f32", 200, 300, 100, "gemm_f32"),
         ("bf16", 300, 64, 256, "gemm_bf16_f32acc"), ("bf16", 20000, 64, 64, "gemm_bf16_f32acc"),
         ("bf16", 512, 512, 256, "gemm_bf16_f32acc"), ("f16", 512, 520, 128, "gemm_f16_f32acc"),
         ("f32", 256, 256, 128, "gemm_tf32_f32acc"), ("f32", 256, 256, 128, "gemm_f32_3xtf32")]


def main():
    torch.cuda.set_device(0)
    data = [inputs.make(M, N, K, dt, "normal", 0.5, seed=i + 1)
            for i, (dt, M, N, K, _) in enumerate(CASES)]
    outs = [None] * len(CASES)
    errors = []
    barrier = threading.Barrier(len(CASES))

    def work(i):
        try:
            dt, M, N, K, entry = CASES[i]
            A, B = data[i]
            a, b = A.cuda(), B.cuda()
            c = torch.full((M, N), float("nan"), device="cuda")
            s = torch.cuda.Stream()
            torch.cuda.synchronize()
            barrier.wait()  # every thread makes its first library call together
            getattr(g14, entry)(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N,
                                s.cuda_stream)
            s.synchronize()
            outs[i] = c.cpu()
        except Exception as e:  # reported below
            errors.append(f"{CASES[i]}: {e!r}")

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(CASES))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    if errors:
        print("\n".join(errors))
        return 1
    assert g14.check_device_error(None) == 0
    bad = []
    for (dt, M, N, K, entry), (A, B), C in zip(CASES, data, outs):
        Ah, Bh = inputs.host_view(A), inputs.host_view(B)
        if entry == "gemm_tf32_f32acc":
            Ah, Bh = oracle.truncate_tf32(Ah), oracle.truncate_tf32(Bh)
        ref, refabs = oracle.gemm(Ah, Bh, dt)
        ok, worst = oracle.within_bound(C.numpy(), ref, refabs, TOL[dt])
        print(f"{entry} {M}x{N}x{K}: worst {worst:.3g}")
        if not ok:
            bad.append(entry)
    return 1 if bad else 0


if __name__ == "__main__":
    sys.exit(main())
