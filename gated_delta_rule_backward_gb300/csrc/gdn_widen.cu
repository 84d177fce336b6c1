// gdn_widen.cu -- 16-bit input storage: widens bf16 / fp16 inputs to fp32.
//
// meTile ("Training kernels and gradients") keeps 16-bit inputs beside fp32 state and
// fp32 gradients.  libgdn takes q, k, v, g, beta and the output cotangent gy stored as
// bf16 or fp16 (gdn_params_t.in_dtype) and widens each into a dense fp32 copy in the
// caller's workspace, exactly (every bf16 and fp16 value is an fp32 value); the fp32
// kernels then run on the copies.  States, checkpoints and every output stay fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

__device__ __forceinline__ float widen(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float widen(__half x) { return __half2float(x); }

// dst[n][t][h][0:D] = src[n s0 + t s1 + h s2 + 0:D], dense fp32.  Rows of D elements; vec:
// every row start is 16-byte aligned and D % 8 == 0 (8 elements per 16-byte load).
template <typename T>
__global__ void __launch_bounds__(256) gdn_widen_kernel(const T* src, long long s0, long long s1, long long s2,
                                                        int N, int Tn, int H, int D, int vec, float* dst)
{
    const long long rows = (long long)N * Tn * H;
    const int per = vec ? D / 8 : D;  // work items per row
    const long long total = rows * per;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long row = idx / per;
        const int e = (int)(idx - row * per);
        const int h = (int)(row % H);
        const long long nt = row / H;
        const int t = (int)(nt % Tn), n = (int)(nt / Tn);
        const T* s = src + n * s0 + t * s1 + h * s2;
        float* d = dst + row * D;
        if (vec) {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(s) + e);
            const T* x = reinterpret_cast<const T*>(&w);
            float4* d4 = reinterpret_cast<float4*>(d) + 2 * e;
            d4[0] = make_float4(widen(x[0]), widen(x[1]), widen(x[2]), widen(x[3]));
            d4[1] = make_float4(widen(x[4]), widen(x[5]), widen(x[6]), widen(x[7]));
        } else {
            d[e] = widen(s[e]);
        }
    }
}

template <typename T>
int launch_t(const void* src, const long long s[3], int N, int Tn, int H, int D, float* dst, cudaStream_t st)
{
    const bool vec = D % 8 == 0 && ((uintptr_t)src % 16) == 0 && s[0] % 8 == 0 && s[1] % 8 == 0 &&
                     s[2] % 8 == 0;
    const long long items = (long long)N * Tn * H * (vec ? D / 8 : D);
    if (items <= 0) return 0;
    long long blocks = (items + 255) / 256;
    if (blocks > 152LL * 16) blocks = 152LL * 16;  // grid-stride: 16 CTAs per SM at most
    gdn_widen_kernel<T><<<(unsigned)blocks, 256, 0, st>>>(static_cast<const T*>(src), s[0], s[1], s[2], N, Tn, H, D,
                                                           vec ? 1 : 0, dst);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_widen(const void* src, int in_dtype, const long long s[3], int N, int Tn, int H, int D, float* dst,
                 void* stream)
{
    cudaStream_t st = (cudaStream_t)stream;
    if (in_dtype == 1) return launch_t<__nv_bfloat16>(src, s, N, Tn, H, D, dst, st);
    if (in_dtype == 2) return launch_t<__half>(src, s, N, Tn, H, D, dst, st);
    return (int)cudaErrorInvalidValue;
}

}  // namespace gdn
