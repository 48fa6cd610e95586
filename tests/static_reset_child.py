"""Child process of tests/test_zz_no_alloc.py::test_static_survives_a_device_reset.

Runs sparse_mla_decode_static, resets the device (which ends the CUDA context whose module
holds the library's scratch array), runs it again, and checks both results against the fp64
oracle and against each other.  Device memory for the inputs and outputs is taken with the
CUDA runtime through ctypes, not through torch: torch keeps device state that a reset would
leave dangling.  torch is used on the CPU only, to build the seeded inputs."""

import ctypes
import sys

import numpy as np

import oracle
import sparse_mla_attention_decode_gb300 as smla
import workloads
from tests.gpu_util import compare


def main() -> int:
    smla.lib()  # loads the library and the CUDA runtime it links
    rt = ctypes.CDLL("libcudart.so.13")
    vp = ctypes.c_void_p
    rt.cudaMalloc.argtypes = [ctypes.POINTER(vp), ctypes.c_size_t]
    rt.cudaMemcpy.argtypes = [vp, vp, ctypes.c_size_t, ctypes.c_int]
    rt.cudaFree.argtypes = [vp]
    H2D, D2H = 1, 2

    def ok(rc, what):
        if rc != 0:
            raise RuntimeError(f"{what}: cuda error {rc}")

    wl = workloads.small(b=6, s_q=1, h_q=128, topk=448, ctx=4096, masked_per_row=40, seed=31)
    q, kv, idx = workloads.to_numpy_inputs(wl)
    q, kv, idx = np.ascontiguousarray(q), np.ascontiguousarray(kv), np.ascontiguousarray(idx)
    b, s_q, h = wl.spec.b, wl.spec.s_q, wl.spec.h_q
    nsm = 16  # several partitions per request: split rows and the combine run
    d = smla.dims_for(b, s_q, h, wl.spec.topk, kv.shape[0])
    ro, rl = oracle.sparse_mla_decode_full(q, kv, idx, wl.sm_scale)

    def run_once():
        bufs = {}
        sizes = {"q": q.nbytes, "kv": kv.nbytes, "idx": idx.nbytes, "out": b * s_q * h * 512 * 2,
                 "lse": b * h * s_q * 4}
        for k, n in sizes.items():
            p = vp()
            ok(rt.cudaMalloc(ctypes.byref(p), n), f"cudaMalloc {k}")
            bufs[k] = p.value
        ok(rt.cudaMemcpy(bufs["q"], q.ctypes.data, q.nbytes, H2D), "copy q")
        ok(rt.cudaMemcpy(bufs["kv"], kv.ctypes.data, kv.nbytes, H2D), "copy kv")
        ok(rt.cudaMemcpy(bufs["idx"], idx.ctypes.data, idx.nbytes, H2D), "copy idx")
        smla.sparse_mla_decode_static(d, nsm, bufs["q"], bufs["kv"], bufs["idx"], wl.sm_scale,
                                      bufs["out"], bufs["lse"], 0)
        rc, word = smla.sparse_mla_static_read_status(d, nsm)
        assert (rc, word) == (0, 0), (rc, word)
        out = np.empty((b, s_q, h, 512), dtype=np.uint16)
        lse = np.empty((b, h, s_q), dtype=np.float32)
        ok(rt.cudaMemcpy(out.ctypes.data, bufs["out"], out.nbytes, D2H), "copy out")
        ok(rt.cudaMemcpy(lse.ctypes.data, bufs["lse"], lse.nbytes, D2H), "copy lse")
        for p in bufs.values():
            ok(rt.cudaFree(p), "cudaFree")
        return out, lse

    def check(out, lse, what):
        o = (out.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        compare(o.reshape(-1, h, 512), lse.astype(np.float64).transpose(0, 2, 1).reshape(-1, h),
                ro.reshape(-1, h, 512), rl.transpose(0, 2, 1).reshape(-1, h), what)

    out1, lse1 = run_once()
    check(out1, lse1, "before the reset")
    ok(rt.cudaDeviceReset(), "cudaDeviceReset")
    out2, lse2 = run_once()
    check(out2, lse2, "after the reset")
    assert np.array_equal(out1, out2) and np.array_equal(lse1.view(np.uint32), lse2.view(np.uint32))
    print("STATIC RESET CHILD OK")
    return 0


if __name__ == "__main__":
    sys.exit(main())
