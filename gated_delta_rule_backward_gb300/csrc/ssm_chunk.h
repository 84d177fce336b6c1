// ssm_chunk.h -- the chunked form of the selective scan with one decay per head (Mamba-2),
// internal to the library: argument block and host entry points used by ssm_scan.cu.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>

namespace ssm {
namespace ssd {

constexpr int kChunk = 64;  // tokens per chunk
constexpr int kP = 64;      // channels per head
constexpr int kS = 128;     // states

struct Args {
    const float *x, *dt, *A, *B, *C, *s0, *ckpt_in, *dy, *dsT;
    float *y, *sT, *ckpt, *ds0, *dx, *ddt, *dB, *dC;
    float *dd, *sin_all, *gvec, *partBC;  // backward workspace
    long long N, T, H, G;
    int K;     // checkpoint interval, a multiple of kChunk
    int n_ck;  // checkpoints (segments) per head
    int nch;   // chunks per sequence
    int m;     // chunks per segment (K / kChunk)
    int HB;    // heads per CTA of the head-blocked kernels
    int nhb;   // such blocks per group
};

// Heads per CTA of the head-blocked kernels: the largest of 4, 2, 1 dividing the heads of a
// group that still leaves at least three CTAs per SM (else 1).
int heads_per_block(long long N, long long nch, long long H, long long G);

struct Workspace {
    size_t dd, sin_all, gvec, partBC, total;
};
Workspace workspace_layout(long long N, long long T, long long H, long long G, int K, int HB);

// Enqueue the forward (y, s_T, checkpoints) or the backward (d_s, dx, ddt, dB, dC) on st;
// the CUDA status of the launches.
int forward(const Args& a, cudaStream_t st);
int backward(const Args& a, cudaStream_t st);

}  // namespace ssd
}  // namespace ssm
