// tv_kv_quantize_q4 / tv_kv_quantize_q3: encode bf16 KV rows in the 4-bit or
// the 3-bit cache format.
//
// The pages pair EAGLE with a quantised KV cache (troisinh.com "EAGLE - Draft
// head ...": an INT4 KV cache leaves room for the draft head; further reading:
// KV-cache quantisation to INT4/INT3).  Format, per row and group of 32 dims:
// fp16 scale and zero, and 4-bit codes two per byte (low nibble = even dim),
// decoding to bf16(fp32(code * scale + zero)).  Encoding in fp32 with IEEE
// rounding at every step:
//   zero = fp16(min x), scale = fp16((max x - min x) / 15), inv = fp32(1 / scale),
//   code = clamp(rint((x - zero) * inv), 0, 15)   (0 when scale is 0).
// The codes are integer decisions taken from floating point: the steps and
// their rounding are part of the format, so they are written out one by one.
// rint of a value clamped to [0, 15] is the low bits of its sum with 1.5 * 2^23
// (the addition rounds to the nearest integer, ties to even).
//
// The 3-bit format has the same parameters with 7 in place of 15 and codes
// 0..7; a row's low two bits of every code come first, four codes per byte
// (byte j: dims 4j .. 4j+3, dim 4j+i in bits 2i and 2i+1), then the third
// bits, eight per byte (byte D/4 + j: dims 8j .. 8j+7, dim 8j+i in bit i).
//
// One thread per group: 64 bytes in (four 16-byte loads), 16 (4-bit) or 12
// (3-bit) bytes of codes and 4 bytes of parameters out; bound by HBM.
#include <cuda_fp16.h>

#include "tv_common.cuh"

namespace tv {

constexpr int kQ4Group = 32;

// The 32 values of group gi, its parameters (scale, zero) as fp16 and the
// fp32 forms used for the codes.
struct GroupEnc {
  float v[kQ4Group];
  __half sh, zh;
  float z, inv;
};
__device__ __forceinline__ void load_group(const uint4* __restrict__ x, int64_t gi, float levels, GroupEnc& g) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = __ldcs(x + gi * 4 + q);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      g.v[q * 8 + 2 * k] = __uint_as_float(u[k] << 16);
      g.v[q * 8 + 2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
    }
  }
  float mn = g.v[0], mx = g.v[0];
#pragma unroll
  for (int k = 1; k < kQ4Group; ++k) {
    mn = fminf(mn, g.v[k]);
    mx = fmaxf(mx, g.v[k]);
  }
  g.zh = __float2half_rn(mn);
  g.sh = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), levels));
  g.z = __half2float(g.zh);
  const float s = __half2float(g.sh);
  // inv = 0 for a constant group: every code is then 0
  g.inv = s > 0.f ? __frcp_rn(s) : 0.f;
}
// code k of the group, clamped to [0, levels]
__device__ __forceinline__ uint32_t group_code(const GroupEnc& g, int k, float levels) {
  const float q = fminf(levels, fmaxf(0.f, __fmul_rn(__fsub_rn(g.v[k], g.z), g.inv)));
  return __float_as_uint(__fadd_rn(q, 12582912.f)) & 15u;
}
__device__ __forceinline__ uint32_t group_params(const GroupEnc& g) {
  return (uint32_t)__half_as_ushort(g.sh) | ((uint32_t)__half_as_ushort(g.zh) << 16);
}

__global__ void __launch_bounds__(256) q4_encode_kernel(const uint4* __restrict__ x, int64_t n_groups,
                                                        uint4* __restrict__ codes, uint32_t* __restrict__ params) {
  griddep_wait();
  const int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gi >= n_groups) return;
  GroupEnc g;
  load_group(x, gi, 15.f, g);
  uint32_t packed[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int k = 0; k < kQ4Group; ++k) packed[k >> 3] |= group_code(g, k, 15.f) << (4 * (k & 7));
  __stcs(codes + gi, make_uint4(packed[0], packed[1], packed[2], packed[3]));
  __stcs(params + gi, group_params(g));
}

// n_per_row groups of 32 dims per row; group gi is group gi % n_per_row of row
// gi / n_per_row, whose codes start at byte (gi / n_per_row) * 12 * n_per_row.
__global__ void __launch_bounds__(256) q3_encode_kernel(const uint4* __restrict__ x, int64_t n_groups,
                                                        int n_per_row, uint32_t* __restrict__ codes,
                                                        uint32_t* __restrict__ params) {
  griddep_wait();
  const int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gi >= n_groups) return;
  GroupEnc g;
  load_group(x, gi, 7.f, g);
  uint32_t lo[2] = {0u, 0u}, hi = 0u;
#pragma unroll
  for (int k = 0; k < kQ4Group; ++k) {
    const uint32_t c = group_code(g, k, 7.f);
    lo[k >> 4] |= (c & 3u) << (2 * (k & 15));
    hi |= (c >> 2) << k;
  }
  const int64_t row = gi / n_per_row;
  const int gr = (int)(gi - row * n_per_row);
  uint32_t* rc = codes + row * 3 * n_per_row;  // the row's 12 * n_per_row bytes as words
  __stcs(rc + 2 * gr, lo[0]);
  __stcs(rc + 2 * gr + 1, lo[1]);
  __stcs(rc + 2 * n_per_row + gr, hi);
  __stcs(params + gi, group_params(g));
}

}  // namespace tv

extern "C" int tv_kv_quantize_q4(const void* x, int64_t rows, int D, uint8_t* codes, void* params, void* stream) {
  tv::clear_error();
  TV_REQUIRE(x && codes && params, TV_ERR_INVALID_ARG, "tv_kv_quantize_q4: NULL pointer");
  TV_REQUIRE(rows >= 0 && D >= tv::kQ4Group && D % tv::kQ4Group == 0 && D <= 1024, TV_ERR_INVALID_ARG,
             "tv_kv_quantize_q4: rows = %lld, D = %d (need D a multiple of 32, at most 1024)", (long long)rows, D);
  TV_REQUIRE(tv::aligned16(x) && tv::aligned16(codes) && (reinterpret_cast<uintptr_t>(params) & 3u) == 0,
             TV_ERR_INVALID_ARG, "tv_kv_quantize_q4: x and codes must be 16-byte aligned, params 4-byte aligned");
  const int64_t n_groups = rows * (D / tv::kQ4Group);
  if (n_groups == 0) return TV_OK;
  const int64_t blocks = (n_groups + 255) / 256;
  TV_REQUIRE(blocks < (1ll << 31), TV_ERR_UNSUPPORTED, "tv_kv_quantize_q4: too many rows");
  TV_CUDA_CHECK(tv::launch_pdl(tv::q4_encode_kernel, dim3((unsigned)blocks), dim3(256), 0, tv::as_stream(stream),
                               reinterpret_cast<const uint4*>(x), n_groups, reinterpret_cast<uint4*>(codes),
                               reinterpret_cast<uint32_t*>(params)));
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}

extern "C" int tv_kv_quantize_q3(const void* x, int64_t rows, int D, uint8_t* codes, void* params, void* stream) {
  tv::clear_error();
  TV_REQUIRE(x && codes && params, TV_ERR_INVALID_ARG, "tv_kv_quantize_q3: NULL pointer");
  TV_REQUIRE(rows >= 0 && D >= tv::kQ4Group && D % tv::kQ4Group == 0 && D <= 1024, TV_ERR_INVALID_ARG,
             "tv_kv_quantize_q3: rows = %lld, D = %d (need D a multiple of 32, at most 1024)", (long long)rows, D);
  TV_REQUIRE(tv::aligned16(x) && (reinterpret_cast<uintptr_t>(codes) & 3u) == 0 &&
                 (reinterpret_cast<uintptr_t>(params) & 3u) == 0,
             TV_ERR_INVALID_ARG, "tv_kv_quantize_q3: x must be 16-byte aligned, codes and params 4-byte aligned");
  const int64_t n_groups = rows * (D / tv::kQ4Group);
  if (n_groups == 0) return TV_OK;
  const int64_t blocks = (n_groups + 255) / 256;
  TV_REQUIRE(blocks < (1ll << 31), TV_ERR_UNSUPPORTED, "tv_kv_quantize_q3: too many rows");
  TV_CUDA_CHECK(tv::launch_pdl(tv::q3_encode_kernel, dim3((unsigned)blocks), dim3(256), 0, tv::as_stream(stream),
                               reinterpret_cast<const uint4*>(x), n_groups, D / tv::kQ4Group,
                               reinterpret_cast<uint32_t*>(codes), reinterpret_cast<uint32_t*>(params)));
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}
