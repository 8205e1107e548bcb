"""The library's host code under sanitizers (CPU only): the CPU side of the CPU/GPU
split attention (bs_cpu_sparse_attn, several std::threads over caller-supplied host
pools and tables) and the host-side checks and sizing, built with AddressSanitizer +
UndefinedBehaviorSanitizer and, separately, ThreadSanitizer, and driven by a small
C++ program over random pools, group sizes 3-5, head_dim 64 and 128, bf16 and fp32,
and a unit with a bad block index and a bad page entry. Numerical agreement with the
oracle is tested in test_split.py; here a clean sanitizer run is the result."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "long_context_serving_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")

HARNESS = r"""
#include <cmath>
#include <cstdio>
#include <cstring>
#include <random>
#include <vector>
#include "bsattn.h"

static uint16_t to_bf16(float f) {
  uint32_t b;
  std::memcpy(&b, &f, 4);
  return uint16_t((b + 0x7fffu + ((b >> 16) & 1u)) >> 16);
}

int main() {
  std::mt19937 rng(7);
  std::normal_distribution<float> nd;
  int fails = 0;
  for (int trial = 0; trial < 6; ++trial) {
    const int B = 2, Hkv = 2, G = (trial % 3) + 3, D = trial % 2 ? 64 : 128, U = B * Hkv;
    const int maxp = 40, n_pages = U * maxp, g = 32, maxsel = 12;
    bs_dims d{};
    d.batch = B; d.n_kv_heads = Hkv; d.n_q_heads = G * Hkv; d.head_dim = D; d.page_size = 16;
    d.max_pages_per_unit = maxp; d.max_blocks_per_unit = 32; d.max_sel_per_unit = maxsel;
    d.max_subs_per_unit = 160; d.max_gather_pages_per_unit = 64; d.n_pages = n_pages;
    d.kv_dtype = trial < 3 ? BS_BF16 : BS_FP32;
    d.q_dtype = d.kv_dtype;
    const size_t el = size_t(n_pages) * 16 * D;
    std::vector<uint16_t> kb(el), vb(el), qb(size_t(B) * d.n_q_heads * D);
    std::vector<float> kf(el), vf(el), qf(qb.size());
    for (size_t i = 0; i < el; ++i) {
      kf[i] = nd(rng); vf[i] = nd(rng); kb[i] = to_bf16(kf[i]); vb[i] = to_bf16(vf[i]);
    }
    for (size_t i = 0; i < qf.size(); ++i) { qf[i] = nd(rng); qb[i] = to_bf16(qf[i]); }
    std::vector<int32_t> pt(size_t(U) * maxp), lens = {600, 17}, gs(U, g), sel(size_t(U) * maxsel, -1), cnt(U);
    for (size_t i = 0; i < pt.size(); ++i) pt[i] = int32_t((i * 7919) % n_pages);
    for (int u = 0; u < U; ++u) {
      const int T = lens[u / Hkv], nb = (T + g - 1) / g;
      int c = 0;
      for (int blk = 0; blk < nb && c < maxsel; blk += 2) sel[size_t(u) * maxsel + c++] = blk;
      if (c < maxsel && sel[size_t(u) * maxsel + c - 1] != nb - 1) sel[size_t(u) * maxsel + c++] = nb - 1;
      cnt[u] = c;
    }
    if (trial == 5) {
      sel[0] = 1000;             // a block past T
      pt[maxp + 1] = n_pages + 5;  // a page outside the pool
    }
    bs_host_kv kv{};
    kv.k_pool = d.kv_dtype == BS_BF16 ? (const void *)kb.data() : (const void *)kf.data();
    kv.v_pool = d.kv_dtype == BS_BF16 ? (const void *)vb.data() : (const void *)vf.data();
    kv.n_pages = n_pages;
    bs_host_tables t{pt.data(), lens.data(), gs.data()};
    std::vector<float> out(size_t(B) * d.n_q_heads * D, NAN), lse(size_t(B) * d.n_q_heads, NAN);
    const void *q = d.q_dtype == BS_BF16 ? (const void *)qb.data() : (const void *)qf.data();
    const bs_status s = bs_cpu_sparse_attn(&d, q, &kv, &t, sel.data(), cnt.data(), out.data(), lse.data(), 3);
    const bs_status want = trial == 5 ? BS_ERR_DEVICE_BOUNDS : BS_OK;
    bool finite = true;
    for (float x : out) finite = finite && std::isfinite(x);
    for (float x : lse) finite = finite && std::isfinite(x);
    if (s != want || !finite) ++fails;

    // Host checks and sizing on the same dims.
    std::vector<int32_t> cls(U, BS_RETRIEVAL), sub(U, 8), k(U, 4), ke(U, 0), sink(U, 32), local(U, 32), rows(U, 160);
    std::vector<int64_t> off(U);
    for (int u = 0; u < U; ++u) off[u] = int64_t(u) * 160 * D;
    bs_head_cfg c{cls.data(), gs.data(), sub.data(), k.data(), ke.data(), sink.data(), local.data(), off.data(),
                  rows.data()};
    if (bs_check_head_cfg(&d, &c, lens.data()) != BS_OK) ++fails;
    if (bs_workspace_size(&d) == 0) ++fails;
    if (std::strcmp(bs_status_string(s), "") == 0) ++fails;
  }
  std::printf("fails %d\n", fails);
  return fails;
}
"""

SANITIZERS = {
    "address+undefined": (["-fsanitize=address", "-fsanitize=undefined", "-fno-omit-frame-pointer"],
                          {"ASAN_OPTIONS": "protect_shadow_gap=0:detect_leaks=1",
                           "UBSAN_OPTIONS": "halt_on_error=1:print_stacktrace=1"}),
    "thread": (["-fsanitize=thread"], {"TSAN_OPTIONS": "halt_on_error=1"}),
}


def _tools():
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    cxx = shutil.which("g++")
    if nvcc is None or cxx is None:
        pytest.skip("needs nvcc and g++")
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")
    if not os.path.exists(os.path.join(cuda_lib, "libcudart_static.a")):
        pytest.skip("needs the static CUDA runtime")
    return nvcc, cxx, cuda_lib


@pytest.mark.parametrize("name", sorted(SANITIZERS))
def test_host_code_under_sanitizer(name, tmp_path):
    nvcc, cxx, cuda_lib = _tools()
    flags, env = SANITIZERS[name]
    objs = []
    for src in ("bs_split.cu", "bs_api.cu"):
        obj = tmp_path / src.replace(".cu", ".o")
        cmd = [nvcc, "-std=c++17", "-O1", "-g", "-gencode", "arch=compute_103a,code=sm_103a", "-I", INCLUDE,
               "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", str(obj)]
        for f in flags:
            cmd += ["-Xcompiler", f]
        subprocess.run(cmd, check=True, capture_output=True)
        objs.append(str(obj))
    harness = tmp_path / "harness.cpp"
    harness.write_text(HARNESS)
    exe = tmp_path / "harness"
    subprocess.run([cxx, "-std=c++17", "-O1", "-g", *flags, "-I", INCLUDE, str(harness), *objs, "-L", cuda_lib,
                    "-lcudart_static", "-ldl", "-lpthread", "-lrt", "-o", str(exe)], check=True, capture_output=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=dict(os.environ, **env), timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "fails 0" in r.stdout
    assert "ERROR" not in r.stderr and "runtime error" not in r.stderr, r.stderr
