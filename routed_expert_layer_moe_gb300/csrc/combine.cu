// Step 5: weighted combine back to token order.
//
// "MoE inference and expert parallelism" (blog.vllbc.top), routing section:
// moe_sum adds the K expert outputs, each weighted by its route weight
// (TopKWeightAndReduce); DeepSeek-V3 Eq. 12 adds the shared expert with
// weight 1.  Summation is in fp32 in the fixed order k = 0..K(+S)-1 and the
// result is rounded once to the output type.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kMaxKS = 33;

// One CTA per (token, chunk of hidden columns); each thread owns VEC columns.
template <typename TY, typename TO, int VEC>
__global__ void __launch_bounds__(128) combine_kernel(const TY* __restrict__ yg, const int32_t* __restrict__ row_of,
                                                      const float* __restrict__ w, TO* __restrict__ out, int H,
                                                      int K, int KS) {
  const int t = blockIdx.x;
  const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * VEC;
  __shared__ int rows[kMaxKS];
  __shared__ float wts[kMaxKS];
  if (threadIdx.x < KS) {
    rows[threadIdx.x] = row_of[(size_t)t * KS + threadIdx.x];
    wts[threadIdx.x] = (threadIdx.x < K) ? w[(size_t)t * K + threadIdx.x] : 1.0f;
  }
  __syncthreads();
  if (c0 >= H) return;
  float acc[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) acc[i] = 0.0f;
  // Up to four rows are requested before their multiply-adds (more bytes in flight per
  // thread); the adds still run in k order, skipping rows that were not placed.
  constexpr int B = 4;
  for (int k0 = 0; k0 < KS; k0 += B) {
    uint4 raw[B];
#pragma unroll
    for (int j = 0; j < B; ++j) {
      const int k = k0 + j;
      if (k < KS && rows[k] >= 0) raw[j] = __ldg(reinterpret_cast<const uint4*>(yg + (size_t)rows[k] * H + c0));
    }
#pragma unroll
    for (int j = 0; j < B; ++j) {
      const int k = k0 + j;
      if (k >= KS || rows[k] < 0) continue;
      const float wk = wts[k];
      if constexpr (sizeof(TY) == 2) {
        static_assert(VEC == 8, "bf16 path reads 16-byte vectors");
        const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(hv[i]);
          acc[2 * i] = fmaf(wk, f.x, acc[2 * i]);
          acc[2 * i + 1] = fmaf(wk, f.y, acc[2 * i + 1]);
        }
      } else {
        static_assert(VEC == 4, "fp32 path reads 16-byte vectors");
        const float4 f = *reinterpret_cast<const float4*>(&raw[j]);
        acc[0] = fmaf(wk, f.x, acc[0]);
        acc[1] = fmaf(wk, f.y, acc[1]);
        acc[2] = fmaf(wk, f.z, acc[2]);
        acc[3] = fmaf(wk, f.w, acc[3]);
      }
    }
  }
  TO* dst = out + (size_t)t * H + c0;
  if constexpr (sizeof(TO) == 2) {
    uint4 raw;
    __nv_bfloat162* hv = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) hv[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    if constexpr (VEC == 8) {
      *reinterpret_cast<uint4*>(dst) = raw;
    } else {
      *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<uint2*>(&raw);
    }
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) dst[i] = acc[i];
  }
}

}  // namespace

int launch_combine(const moe_problem& p, const void* yg, const int32_t* row_of, const float* w, void* out,
                   cudaStream_t st) {
  if (p.T == 0) return MOE_OK;
  const int KS = p.K + p.has_shared;
  const int threads = 128;
  if (p.wt == MOE_F32) {
    const dim3 grid(p.T, (p.H / 4 + threads - 1) / threads);
    combine_kernel<float, float, 4><<<grid, threads, 0, st>>>((const float*)yg, row_of, w, (float*)out, p.H, p.K,
                                                               KS);
  } else {
    const dim3 grid(p.T, (p.H / 8 + threads - 1) / threads);
    combine_kernel<__nv_bfloat16, __nv_bfloat16, 8><<<grid, threads, 0, st>>>(
        (const __nv_bfloat16*)yg, row_of, w, (__nv_bfloat16*)out, p.H, p.K, KS);
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
