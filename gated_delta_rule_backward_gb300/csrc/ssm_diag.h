// ssm_diag.h -- the selective scan with one decay per state (Mamba-1: one channel a head, 16
// states) split by checkpoint segments, internal to the library: argument block and host entry
// points used by ssm_scan.cu.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>

namespace ssm {
namespace diag {

constexpr int kS = 16;   // states
constexpr int kSB = 32;  // tokens per sub-block of the backward

struct Args {
    const float *x, *dt, *A, *B, *C, *s0, *ckpt_in, *dy, *dsT;
    float *y, *sT, *ckpt, *ds0, *dx, *ddt, *dB, *dC;
    float *sin_sb, *U, *Gb, *carry, *partBC;  // backward workspace
    long long N, T, H, G;
    int K;     // checkpoint interval (segment length)
    int n_ck;  // segments per sequence
    int spk;   // sub-blocks per segment, ceil(K / kSB)
    int nsb;   // sub-blocks per sequence, n_ck spk
    int nbg;   // blocks of 16 channels per group
};

struct Workspace {
    size_t sin_sb, U, Gb, carry, partBC, total;
};
Workspace workspace_layout(long long N, long long T, long long H, long long G, int K);

int forward(const Args& a, cudaStream_t st);
int backward(const Args& a, cudaStream_t st);

}  // namespace diag
}  // namespace ssm
