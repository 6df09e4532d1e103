// CUDA-core fp32 GEMMs of the sampler: the logits y = (H . E^T) / T, the self-conditioning
// partials O = exp(y - m) . E over vocabulary splits, and the hidden-state stand-in
// H = bf16(tanh(W . [bf16(s); E[x]])). They serve fp32 inputs (which the bf16 tensor cores
// cannot take exactly) and act as the CUDA-core cross-check of the tensor-core kernels.
//
// Definitions: DiffusionGemma Technical Report, section 6 "Sampling" (softmax over the full
// vocabulary and the self-conditioning embedding matmul).
#include <cuda_bf16.h>

#include <algorithm>

#include "ds_internal.h"

namespace ds {
namespace {

constexpr int BM = 128, BK = 16, THREADS = 256;

DS_DEV float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

template <bool FP32>
DS_DEV float load_elem(const void* p, size_t idx) {
  if constexpr (FP32) {
    return static_cast<const float*>(p)[idx];
  } else {
    return bf16_to_f32(static_cast<const uint16_t*>(p)[idx]);
  }
}

// C[M, N] = A[M, K] . B[N, K]^T with both operands K-contiguous; 128 x BN tiles, 8 x (BN/16)
// outputs per thread. Requires M % 128 == 0, N % BN == 0, K % 16 == 0.
template <int BN, class LoadA, class LoadB, class Epi>
DS_DEV void gemm_nt_tile(int m0, int n0, int K, LoadA la, LoadB lb, Epi epi) {
  constexpr int TN = BN / 16;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[8][TN];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int c = 0; c < TN; ++c) acc[a][c] = 0.f;
  for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
    for (int q = 0; q < (BM * BK) / THREADS; ++q) {
      const int e = threadIdx.x + THREADS * q;
      As[e % BK][e / BK] = la(m0 + e / BK, k0 + e % BK);
    }
#pragma unroll
    for (int q = 0; q < (BN * BK) / THREADS; ++q) {
      const int e = threadIdx.x + THREADS * q;
      Bs[e % BK][e / BK] = lb(n0 + e / BK, k0 + e % BK);
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[8], b[TN];
#pragma unroll
      for (int q = 0; q < 8; ++q) a[q] = As[kk][ty + 16 * q];
#pragma unroll
      for (int q = 0; q < TN; ++q) b[q] = Bs[kk][tx + 16 * q];
#pragma unroll
      for (int p = 0; p < 8; ++p)
#pragma unroll
        for (int q = 0; q < TN; ++q) acc[p][q] = fmaf(a[p], b[q], acc[p][q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int p = 0; p < 8; ++p)
#pragma unroll
    for (int q = 0; q < TN; ++q) epi(m0 + ty + 16 * p, n0 + tx + 16 * q, acc[p][q]);
}

template <bool FP32>
__global__ void __launch_bounds__(THREADS) k_logits_simt(const void* __restrict__ H,
                                                         const void* __restrict__ E, int64_t V,
                                                         int d, int L, const float* __restrict__ T,
                                                         const uint8_t* __restrict__ done,
                                                         float* __restrict__ Y) {
  const int m0 = blockIdx.y * BM;
  const int n0 = blockIdx.x * 128;
  const int b = m0 / L;
  if (done && done[b]) return;
  const float invT = 1.0f / T[b];
  gemm_nt_tile<128>(
      m0, n0, d, [&](int m, int k) { return load_elem<FP32>(H, (size_t)m * d + k); },
      [&](int n, int k) { return load_elem<FP32>(E, (size_t)n * d + k); },
      [&](int m, int n, float acc) { Y[(size_t)m * V + n] = acc * invT; });
}

// O_part[s][m, n] = sum over the split's tokens j of (hi + lo)[m, j] * E[j, n].
template <bool FP32>
__global__ void __launch_bounds__(THREADS) k_selfcond_simt(const uint16_t* __restrict__ Phi,
                                                           const uint16_t* __restrict__ Plo,
                                                           const void* __restrict__ E, int64_t V,
                                                           int d, int R, int L,
                                                           const uint8_t* __restrict__ done,
                                                           int64_t kb_per_split,
                                                           float* __restrict__ Opart) {
  constexpr int BN = 64, TN = BN / 16;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN, split = blockIdx.z;
  if (done && done[m0 / L]) return;
  const int64_t j_begin = (int64_t)split * kb_per_split * BK;
  const int64_t j_end = min(V, j_begin + kb_per_split * BK);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[8][TN];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int c = 0; c < TN; ++c) acc[a][c] = 0.f;
  for (int64_t k0 = j_begin; k0 < j_end; k0 += BK) {
#pragma unroll
    for (int q = 0; q < (BM * BK) / THREADS; ++q) {
      const int e = threadIdx.x + THREADS * q;
      const size_t at = (size_t)(m0 + e / BK) * V + (size_t)(k0 + e % BK);
      As[e % BK][e / BK] = bf16_to_f32(Phi[at]) + bf16_to_f32(Plo[at]);
    }
#pragma unroll
    for (int q = 0; q < (BN * BK) / THREADS; ++q) {
      const int e = threadIdx.x + THREADS * q;
      Bs[e / BN][e % BN] = load_elem<FP32>(E, (size_t)(k0 + e / BN) * d + n0 + e % BN);
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[8], b[TN];
#pragma unroll
      for (int q = 0; q < 8; ++q) a[q] = As[kk][ty + 16 * q];
#pragma unroll
      for (int q = 0; q < TN; ++q) b[q] = Bs[kk][tx + 16 * q];
#pragma unroll
      for (int p = 0; p < 8; ++p)
#pragma unroll
        for (int q = 0; q < TN; ++q) acc[p][q] = fmaf(a[p], b[q], acc[p][q]);
    }
    __syncthreads();
  }
  float* out = Opart + (size_t)split * R * d;
#pragma unroll
  for (int p = 0; p < 8; ++p)
#pragma unroll
    for (int q = 0; q < TN; ++q) out[(size_t)(m0 + ty + 16 * p) * d + n0 + tx + 16 * q] = acc[p][q];
}

// A canvas token outside [0, V) is a caller error that no host check can see in a device
// buffer: the row read is clamped into E (so no access leaves it) and kErrBounds is recorded in
// the device error word (ds_sampler_device_status -> DS_ERR_DEVICE).
DS_DEV int64_t checked_token(int32_t t, int64_t V, uint32_t* err) {
  if (t >= 0 && (int64_t)t < V) return t;
  atomicOr(err, kErrBounds);
  return t < 0 ? 0 : V - 1;
}

__global__ void __launch_bounds__(THREADS) k_standin_simt(const uint16_t* __restrict__ W,
                                                          const float* __restrict__ s_prev,
                                                          const uint16_t* __restrict__ E,
                                                          const int32_t* __restrict__ canvas,
                                                          const uint8_t* __restrict__ done, int d,
                                                          int L, int64_t V, uint32_t* err,
                                                          uint16_t* __restrict__ H) {
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * 64;
  if (done && done[m0 / L]) return;
  gemm_nt_tile<64>(
      m0, n0, 2 * d,
      [&](int m, int k) {
        if (k < d) return __bfloat162float(__float2bfloat16_rn(s_prev[(size_t)m * d + k]));
        return bf16_to_f32(E[(size_t)checked_token(canvas[m], V, err) * d + (k - d)]);
      },
      [&](int n, int k) { return bf16_to_f32(W[(size_t)n * 2 * d + k]); },
      [&](int m, int n, float acc) {
        H[(size_t)m * d + n] = __bfloat16_as_ushort(__float2bfloat16_rn(tanhf(acc)));
      });
}

// U[r, k] = k < d ? bf16(s_prev[r, k]) : E[canvas[r], k - d], eight bf16 per thread.
__global__ void k_standin_gather(const float* __restrict__ s_prev, const uint16_t* __restrict__ E,
                                 const int32_t* __restrict__ canvas,
                                 const uint8_t* __restrict__ done, int R, int d, int L, int64_t V,
                                 uint32_t* err, uint16_t* __restrict__ U) {
  const int per_row = (2 * d) / 8;
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < (int64_t)R * per_row;
       q += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(q / per_row), k = (int)(q % per_row) * 8;
    if (done && done[r / L]) continue;
    uint4 out;
    if (k < d) {
      const float4 a = *reinterpret_cast<const float4*>(s_prev + (size_t)r * d + k);
      const float4 b = *reinterpret_cast<const float4*>(s_prev + (size_t)r * d + k + 4);
      const __nv_bfloat162 h0 = __floats2bfloat162_rn(a.x, a.y), h1 = __floats2bfloat162_rn(a.z, a.w);
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(b.x, b.y), h3 = __floats2bfloat162_rn(b.z, b.w);
      out = make_uint4(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1),
                       *reinterpret_cast<const uint32_t*>(&h2), *reinterpret_cast<const uint32_t*>(&h3));
    } else {
      out = *reinterpret_cast<const uint4*>(E + (size_t)checked_token(canvas[r], V, err) * d +
                                            (k - d));
    }
    *reinterpret_cast<uint4*>(U + (size_t)r * 2 * d + k) = out;
  }
}

}  // namespace

void launch_standin_gather(const float* s_prev, const uint16_t* E, const int32_t* canvas,
                           const uint8_t* done, int R, int d, int L, int64_t V, uint32_t* err,
                           uint16_t* U, cudaStream_t st) {
  const int64_t n = (int64_t)R * (2 * d) / 8;
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, 4096);
  k_standin_gather<<<blocks, 256, 0, st>>>(s_prev, E, canvas, done, R, d, L, V, err, U);
}

void launch_logits_simt(const void* H, const void* E, bool fp32_inputs, int R, int64_t V, int d,
                        int L, const float* T, const uint8_t* done, float* Y, cudaStream_t st) {
  const dim3 grid((unsigned)(V / 128), (unsigned)(R / BM));
  if (fp32_inputs)
    k_logits_simt<true><<<grid, THREADS, 0, st>>>(H, E, V, d, L, T, done, Y);
  else
    k_logits_simt<false><<<grid, THREADS, 0, st>>>(H, E, V, d, L, T, done, Y);
}

void launch_selfcond_simt(const uint16_t* Phi, const uint16_t* Plo, const void* E,
                          bool fp32_inputs, int R, int64_t V, int d, int L, const uint8_t* done,
                          int S, float* Opart, cudaStream_t st) {
  const int64_t nkb = V / BK;
  const int64_t per = (nkb + S - 1) / S;
  const dim3 grid((unsigned)(d / 64), (unsigned)(R / BM), (unsigned)S);
  if (fp32_inputs)
    k_selfcond_simt<true><<<grid, THREADS, 0, st>>>(Phi, Plo, E, V, d, R, L, done, per, Opart);
  else
    k_selfcond_simt<false><<<grid, THREADS, 0, st>>>(Phi, Plo, E, V, d, R, L, done, per, Opart);
}

void launch_standin_simt(const uint16_t* W, const float* s_prev, const uint16_t* E,
                         const int32_t* canvas, const uint8_t* done, int R, int d, int L,
                         int64_t V, uint32_t* err, uint16_t* H_out, cudaStream_t st) {
  const dim3 grid((unsigned)(d / 64), (unsigned)(R / BM));
  k_standin_simt<<<grid, THREADS, 0, st>>>(W, s_prev, E, canvas, done, d, L, V, err, H_out);
}

}  // namespace ds
