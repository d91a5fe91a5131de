"""GPU: the C ABI driven from a plain C program, with no PyTorch.

A C99 program allocates device memory with the CUDA runtime, runs one
verify and one commit through ``include/kda.h`` on a one-token case whose
result has a closed form, and checks it:
  - zero checkpoint, q = k = all ones, v[r] = (r - 64) / 64, g_raw = 0,
    g_bias = 0, A_log = 0 (so the decay is 1/2, irrelevant on a zero state),
    beta_raw = 0 (beta = 1/2), one head, window 1;
  - the state after the token is S' = beta v k^T with k^ = k / sqrt(128 +
    1e-6), and the output o = S' q^ = beta v (k^ . q^) with
    q^ = q scale / sqrt(128 + 1e-6);
  - the verify writes o (bf16) and stores no state; the commit (one token
    accepted) writes S' to the row's slot and leaves the null slot at zero.
"""

import os
import shutil
import subprocess

import pytest

from linear_attention_speculative_kda_gb300 import build as kbuild

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")

PROGRAM = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "kda.h"

#define D 128
#define CHECK(x) do { if ((x) != cudaSuccess) { printf("cuda error line %d\n", __LINE__); return 20; } } while (0)

static uint16_t bf16_of(float f) {  /* round to nearest even */
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float float_of(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

int main(void) {
    const int S = 2, R = 1, Q = 1, H = 1;
    uint16_t hq[D], hk[D], hv[D], hg[D], hbeta = bf16_of(0.0f);
    float hA = 0.0f, hbias[D], state[2 * D * D];
    int32_t hcu[2] = {0, 1}, hslot[1] = {1}, hacc[1] = {1}, herr = 0;
    uint16_t hout[D];
    int r, c;
    for (r = 0; r < D; ++r) {
        hq[r] = bf16_of(1.0f);
        hk[r] = bf16_of(1.0f);
        hv[r] = bf16_of((float)(r - 64) / 64.0f);
        hg[r] = bf16_of(0.0f);
        hbias[r] = 0.0f;
    }
    void *dq, *dk, *dv, *dg, *dbeta, *drec, *dout;
    float *dA, *dbias, *dpool;
    int32_t *dcu, *dslot, *dacc, *derr;
    size_t rec_bytes = kda_records_bytes(H, Q, R);
    if (rec_bytes == 0) return 1;
    CHECK(cudaMalloc(&dq, sizeof hq)); CHECK(cudaMalloc(&dk, sizeof hk));
    CHECK(cudaMalloc(&dv, sizeof hv)); CHECK(cudaMalloc(&dg, sizeof hg));
    CHECK(cudaMalloc(&dbeta, sizeof hbeta)); CHECK(cudaMalloc(&drec, rec_bytes));
    CHECK(cudaMalloc(&dout, sizeof hout)); CHECK(cudaMalloc((void **)&dA, sizeof hA));
    CHECK(cudaMalloc((void **)&dbias, sizeof hbias));
    CHECK(cudaMalloc((void **)&dpool, sizeof state));
    CHECK(cudaMalloc((void **)&dcu, sizeof hcu)); CHECK(cudaMalloc((void **)&dslot, sizeof hslot));
    CHECK(cudaMalloc((void **)&dacc, sizeof hacc)); CHECK(cudaMalloc((void **)&derr, sizeof herr));
    CHECK(cudaMemcpy(dq, hq, sizeof hq, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(dk, hk, sizeof hk, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(dv, hv, sizeof hv, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(dg, hg, sizeof hg, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(dbeta, &hbeta, sizeof hbeta, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(dA, &hA, sizeof hA, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(dbias, hbias, sizeof hbias, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(dcu, hcu, sizeof hcu, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(dslot, hslot, sizeof hslot, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(dacc, hacc, sizeof hacc, cudaMemcpyHostToDevice));
    CHECK(cudaMemset(dpool, 0, sizeof state));
    CHECK(cudaMemset(derr, 0, sizeof herr));

    kda_config cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.num_heads = H; cfg.head_dim = D; cfg.window = Q; cfg.num_slots = S;
    cfg.record_slots = R; cfg.use_lower_bound = 0; cfg.scale = 1.0f / sqrtf((float)D);
    cfg.stride_q_t = cfg.stride_k_t = cfg.stride_v_t = cfg.stride_g_t = H * D;
    cfg.stride_beta_t = H; cfg.record_format = KDA_RECORDS_RAW;

    if (kda_verify(&cfg, dq, dk, dv, dg, dbeta, dA, dbias, dpool, dcu, dslot, 1, NULL, NULL,
                   drec, dout, NULL, derr, NULL) != KDA_OK) return 2;
    CHECK(cudaDeviceSynchronize());
    CHECK(cudaMemcpy(hout, dout, sizeof hout, cudaMemcpyDeviceToHost));
    CHECK(cudaMemcpy(state, dpool, sizeof state, cudaMemcpyDeviceToHost));
    for (r = 0; r < 2 * D * D; ++r)
        if (state[r] != 0.0f) return 3;  /* the verify stores no state */

    const double kk = 1.0 / sqrt(128.0 + 1e-6);
    const double qq = (1.0 / sqrt(128.0)) / sqrt(128.0 + 1e-6);
    for (r = 0; r < D; ++r) {
        const double v = (double)(r - 64) / 64.0;
        const double o = 0.5 * v * (128.0 * kk * qq);
        if (fabs((double)float_of(hout[r]) - o) > fabs(o) / 256.0 + 1e-7) {
            printf("out[%d] = %g, want %g\n", r, (double)float_of(hout[r]), o);
            return 4;
        }
    }

    if (kda_commit(&cfg, dA, dbias, dpool, dcu, dslot, 1, dacc, NULL, drec, NULL, NULL, derr,
                   NULL) != KDA_OK) return 5;
    CHECK(cudaDeviceSynchronize());
    CHECK(cudaMemcpy(state, dpool, sizeof state, cudaMemcpyDeviceToHost));
    CHECK(cudaMemcpy(&herr, derr, sizeof herr, cudaMemcpyDeviceToHost));
    if (herr != 0) return 6;
    for (r = 0; r < D * D; ++r)
        if (state[r] != 0.0f) return 7;  /* the null slot stays zero */
    for (r = 0; r < D; ++r)
        for (c = 0; c < D; ++c) {
            const double want = 0.5 * ((double)(r - 64) / 64.0) * kk;
            const double got = state[D * D + r * D + c];
            if (fabs(got - want) > 1e-6 * fabs(want) + 1e-9) {
                printf("state[%d][%d] = %g, want %g\n", r, c, got, want);
                return 8;
            }
        }
    printf("ok\n");
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_verify_and_commit(tmp_path):
    lib = kbuild.build()
    libdir = os.path.dirname(lib)
    src = tmp_path / "kda_from_c.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "kda_from_c"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O2",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
                    str(src), "-L", libdir, "-lkda", f"-Wl,-rpath,{libdir}",
                    "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-lm", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
    assert out.stdout.strip() == "ok"
