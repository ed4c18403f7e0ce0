"""The debug build (lib/libgemm_gb300_debug.so, -DGEMM_DEBUG) on small in-bounds shapes.

In that build every kernel checks the global indices it computes against the extents of
its operands before each access; a failed check raises a flag (gemm_get_device_status
then returns GEMM_ERR_DEVICE_BOUNDS) and the access is skipped.  On correct shapes no
check may fail and the results must be those of the release build: exact on
integer-valued inputs.  Every kernel family runs once, in a fresh process with
GEMM_GB300_DEBUG=1 (the variable selects the library when the package is imported).
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import numpy as np, torch
import oracle, seeded_inputs as si
import programming_tiled_gemm_gb300 as g
assert g.DEBUG and g.LIB_PATH.endswith("libgemm_gb300_debug.so")
lib = g.Gemm(0)
dev = torch.device("cuda")
ran = []

def check(name, got, ref):
    torch.cuda.synchronize()
    st = lib.device_status()
    assert st == g.GEMM_OK, (name, g.status_string(st))
    got = got.cpu().double().numpy() if isinstance(got, torch.Tensor) else got
    assert np.array_equal(got, ref), (name, np.abs(got - ref).max())
    ran.append(name)

# fp32 kernels: tiled 128x256 (split-K and last-wave slices), tiled 64x128, skinny in
# registers and through a TMA ring, the persistent kernel (auto and forced split)
for kernel, split, (M, N, K) in [(1, 0, (300, 600, 200)), (1, 3, (300, 600, 200)), (1, 0, (1664, 3328, 512)),
                                 (2, 0, (60, 300, 130)), (3, 0, (20, 1030, 300)), (3, 4, (20, 1030, 300)),
                                 (4, 0, (16, 1024, 700)), (5, 0, (300, 600, 200)), (5, 0, (1664, 3328, 512)),
                                 (5, 3, (130, 260, 300))]:
    lib.set_option(g.GEMM_OPT_F32_KERNEL, kernel)
    lib.set_option(g.GEMM_OPT_SPLIT_K, split)
    A, B = si.integer_copy(M, N, K, seed=M + N + K)
    check("f32 kernel %d split %d %s" % (kernel, split, (M, N, K)), lib.matmul(A.to(dev), B.to(dev)),
          oracle.gemm(A.numpy(), B.numpy()))
lib.set_option(g.GEMM_OPT_F32_KERNEL, 0)
lib.set_option(g.GEMM_OPT_SPLIT_K, 0)

# fp32 product with bf16 output through the epilogue pass (small integers: exact in bf16)
A, B = si.integer_copy(70, 90, 8, seed=5)
C = torch.empty((70, 90), dtype=torch.bfloat16, device=dev)
lib.matmul(A.to(dev), B.to(dev), out=C, alpha=0.5)
check("f32 -> bf16 epilogue", C.float(), 0.5 * oracle.gemm(A.numpy(), B.numpy()))

# tensor-core kernels: CTA pairs (last wave cut along K), single CTA, K split over a cluster
for pair, (M, N, K) in [(2, (520, 264, 136)), (0, (1024, 2048, 4096)), (1, (300, 264, 72)), (0, (100, 1000, 1104))]:
    lib.set_option(g.GEMM_OPT_TC_PAIR, pair)
    A, B = si.integer_copy(M, N, K, seed=M + 1, dtype="bf16")
    check("bf16 pair option %d %s" % (pair, (M, N, K)), lib.matmul(A.to(dev), B.to(dev)),
          oracle.gemm(A.float().numpy(), B.float().numpy()))
lib.set_option(g.GEMM_OPT_TC_PAIR, 0)

# convolution: im2col, implicit GEMM, tensor cores (channel-last bf16, then channel-first)
gen = si.generator(7)
x = si.ints((3, 6, 5, 7, 12), gen).float()
w = si.ints((4, 3, 2, 1, 3, 5), gen).float()
check("im2col", lib.im2col4d(x.to(dev), [2, 1, 3, 5]), oracle.im2col4d(x.numpy(), (2, 1, 3, 5)))
check("conv implicit", lib.conv4d_implicit(x.to(dev), w.to(dev)), oracle.conv4d_direct(x.numpy(), w.numpy()))
gen = si.generator(8)
x = si.ints((16, 8, 8, 8, 8), gen).float()
w = si.ints((32, 16, 3, 3, 3, 3), gen).float()
xc, wc = si.channel_last(x, w, "bf16")
ref = np.ascontiguousarray(np.moveaxis(oracle.conv4d_direct(x.numpy(), w.numpy()), 0, -1))
check("conv tensor cores", lib.conv4d_cl(xc.to(dev), wc.to(dev)), ref)
gen = si.generator(9)
x = si.ints((3, 6, 5, 7, 12), gen).float()
w = si.ints((16, 3, 2, 1, 3, 5), gen).float()
check("conv tensor cores, channel-first", lib.conv4d_tc(x.to(torch.bfloat16).to(dev), w.to(torch.bfloat16).to(dev)),
      oracle.conv4d_direct(x.numpy(), w.numpy()))
lib.close()
print("debug build ok:", len(ran), "products")
"""


def test_debug_build_runs_every_kernel_family_without_a_failed_check():
    import __graft_entry__
    __graft_entry__.build()
    env = dict(os.environ, GEMM_GB300_DEBUG="1", PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    p = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True, env=env, cwd=ROOT, timeout=900)
    assert p.returncode == 0, p.stdout + p.stderr
    assert "debug build ok: 19 products" in p.stdout, p.stdout + p.stderr
