// Row-wise fused kernels of the decoder, one CTA per action-chunk row.
//
// row_kernel: the consumer of a K-split GEMM (blog post "Embodied inference
// acceleration", section "Static quantisation": gated residual + AdaRMSNorm +
// FP8 convert fused, with the next layer's condition parameters, emitting exactly
// the operand the next GEMM reads). It sums the partial planes in fixed order,
// dequantises with fp32(s_a * s_w), applies the gated residual
// x <- x + gate * y, then (optionally) the flow-matching step boundary
// (final AdaRMSNorm * gamma_f, output projection, Euler update of the action
// chunk, input projection of the next step) and finally
// q = Q(x / sqrt(mean(x^2) + eps) * (1 + scale) + shift) (blog post, "CUDA
// Graph vs graph simplification": the input-dependent RMS stays, gamma is folded
// into the next GEMM's weights). The row statistic uses warp shuffles and one
// shared-memory exchange.
//
// Create-time kernels: timestep embedding and the per-step modulation table.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace fm {

namespace {

constexpr int kRowThreads = 256;
constexpr int kMaxA = 32;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();   // protect red[] from a previous use
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) t += red[w];
  return t;
}

__device__ __forceinline__ uint8_t e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ void store_q4(void* q, size_t idx, float4 h, int fp8, float rs) {
  if (fp8 == kQFp8AsF16) {   // E4M3 codes stored as their f16 values (exact)
    const uint8_t c[4] = {e4m3(h.x * rs), e4m3(h.y * rs), e4m3(h.z * rs), e4m3(h.w * rs)};
    __half v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c[i]), __NV_E4M3));
    uint2 u;
    u.x = static_cast<uint32_t>(__half_as_ushort(v[0])) | (static_cast<uint32_t>(__half_as_ushort(v[1])) << 16);
    u.y = static_cast<uint32_t>(__half_as_ushort(v[2])) | (static_cast<uint32_t>(__half_as_ushort(v[3])) << 16);
    *reinterpret_cast<uint2*>(static_cast<__half*>(q) + idx) = u;
  } else if (fp8) {
    uchar4 c;
    c.x = e4m3(h.x * rs);
    c.y = e4m3(h.y * rs);
    c.z = e4m3(h.z * rs);
    c.w = e4m3(h.w * rs);
    *reinterpret_cast<uchar4*>(static_cast<uint8_t*>(q) + idx) = c;
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(h.x, h.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(h.z, h.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(q) + idx) = u;
  }
}

__global__ void __launch_bounds__(kRowThreads) row_kernel(const RowArgs r) {
  extern __shared__ float xs[];   // the row, N floats
  __shared__ float red[kRowThreads / 32];
  __shared__ float sa_vec[kMaxA];
  __shared__ float vred[kRowThreads / 32][kMaxA];

  const int m = blockIdx.x;
  const int tid = threadIdx.x;
  const int N = r.N;
  const int n4 = N / 4;
  const bool tl_on = r.tl != nullptr && tid == 0;   // diagnostic timeline: entry, after the wait, exit
  __shared__ uint64_t tt[kTlStamps];   // timeline stamps (thread 0)
  if (tl_on)
    for (int i = 0; i < kTlStamps; ++i) tt[i] = 0;
  if (tl_on) tt[0] = global_ns();
  if (r.stamp_kind == 1 && m == 0 && tid == 0) {   // the decision's first kernel starts
    r.stamp[0] = global_ns();
    r.stamp[1] = 0ull;
  }
  pdl_trigger();
  // Per-create constants (scales, modulation rows) do not depend on the previous
  // kernel: fetch them before waiting for it.
  const float ds = r.parts ? __fmul_rn(*r.sa, *r.sw) : 0.f;
  // E4M3: the reciprocal of the static scale; four-bit: the tensor scale itself
  const float rs_q = (r.do_quant && r.q_fp8) ? (r.q_fp8 == kQNvfp4AsF16 ? *r.sq : 1.0f / *r.sq) : 1.0f;
  constexpr int kPre = 2;   // column groups per thread kept in registers (N <= 2048); the
                            // selects below name both explicitly (static register indices)
  float4 gate_v[kPre], scale_v[kPre], shift_v[kPre];
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    const int c = tid + u * kRowThreads;
    if (c < n4) {
      if (r.gate) gate_v[u] = *reinterpret_cast<const float4*>(r.gate + c * 4);
      if (r.do_quant) {
        scale_v[u] = *reinterpret_cast<const float4*>(r.scale + c * 4);
        shift_v[u] = *reinterpret_cast<const float4*>(r.shift + c * 4);
      }
    }
  }
  pdl_wait();
  if (tl_on) tt[1] = global_ns();

  float* xrow = r.x + static_cast<size_t>(m) * N;
  const float* xin = r.x_src ? r.x_src + static_cast<size_t>(m) * N : xrow;
  const size_t plane = static_cast<size_t>(r.M) * N;

  // ---- residual update (skipped when the step head recomputes x from the actions)
  float ss = 0.f;
  const bool load_x = r.parts || r.x_src || !r.do_head || r.do_tail;
  for (int c = tid; load_x && c < n4; c += kRowThreads) {
    float4 x = *reinterpret_cast<const float4*>(xin + c * 4);
    if (r.parts) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      // planes in groups of four, each group's loads issued together (slots past the
      // last plane re-read the group's first and are dropped); summed in plane order
      for (int p0 = 0; p0 < r.nparts; p0 += 4) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int p = p0 + j < r.nparts ? p0 + j : p0;
          v[j] = *reinterpret_cast<const float4*>(r.parts + p * plane + static_cast<size_t>(m) * N + c * 4);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (p0 + j < r.nparts) {
            acc.x += v[j].x;
            acc.y += v[j].y;
            acc.z += v[j].z;
            acc.w += v[j].w;
          }
        }
      }
      float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r.bias) b = *reinterpret_cast<const float4*>(r.bias + c * 4);
      const int u = (c - tid) / kRowThreads;
      const float4 gt = u == 0 ? gate_v[0] : u == 1 ? gate_v[1] : *reinterpret_cast<const float4*>(r.gate + c * 4);
      x.x = fmaf(gt.x, fmaf(acc.x, ds, b.x), x.x);
      x.y = fmaf(gt.y, fmaf(acc.y, ds, b.y), x.y);
      x.z = fmaf(gt.z, fmaf(acc.z, ds, b.z), x.z);
      x.w = fmaf(gt.w, fmaf(acc.w, ds, b.w), x.w);
    }
    *reinterpret_cast<float4*>(xs + c * 4) = x;
    if (!r.do_head && (r.parts || r.x_src)) *reinterpret_cast<float4*>(xrow + c * 4) = x;
    ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
  }

  // ---- Euler step tail: a <- a + dt * (AdaRMSNorm_f(x) * gamma_f . w_out^T + b_out)
  if (r.do_tail) {
    const float rr = rsqrtf(block_sum(ss, red) / N + r.eps);
    float acc[kMaxA];
#pragma unroll
    for (int a = 0; a < kMaxA; ++a) acc[a] = 0.f;
    for (int c = tid; c < n4; c += kRowThreads) {
      const float4 x = *reinterpret_cast<const float4*>(xs + c * 4);
      const float4 sc = *reinterpret_cast<const float4*>(r.scale_f + c * 4);
      const float4 sh = *reinterpret_cast<const float4*>(r.shift_f + c * 4);
      const float4 gf = *reinterpret_cast<const float4*>(r.gamma_f + c * 4);
      float hf[4];
      hf[0] = fmaf(x.x * rr, 1.f + sc.x, sh.x) * gf.x;
      hf[1] = fmaf(x.y * rr, 1.f + sc.y, sh.y) * gf.y;
      hf[2] = fmaf(x.z * rr, 1.f + sc.z, sh.z) * gf.z;
      hf[3] = fmaf(x.w * rr, 1.f + sc.w, sh.w) * gf.w;
      // all A weight loads first (rows past A re-read row 0 and are dropped): loads
      // under a per-row branch would each wait for the previous one's FMAs
      uint2 wv[kMaxA];
#pragma unroll
      for (int a = 0; a < kMaxA; ++a)
        wv[a] = *reinterpret_cast<const uint2*>(r.w_out + static_cast<size_t>(a < r.A ? a : 0) * N + c * 4);
#pragma unroll
      for (int a = 0; a < kMaxA; ++a) {
        const __nv_bfloat162 w01 = *reinterpret_cast<const __nv_bfloat162*>(&wv[a].x);
        const __nv_bfloat162 w23 = *reinterpret_cast<const __nv_bfloat162*>(&wv[a].y);
        acc[a] = fmaf(hf[0], __low2float(w01), acc[a]);
        acc[a] = fmaf(hf[1], __high2float(w01), acc[a]);
        acc[a] = fmaf(hf[2], __low2float(w23), acc[a]);
        acc[a] = fmaf(hf[3], __high2float(w23), acc[a]);
      }
    }
    const int warp = tid >> 5, lane = tid & 31;
#pragma unroll
    for (int a = 0; a < kMaxA; ++a) {
      float v = acc[a];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) vred[warp][a] = v;
    }
    __syncthreads();
    if (tid < r.A) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kRowThreads / 32; ++w) v += vred[w][tid];
      float* arow = r.a + static_cast<size_t>(m) * r.A;
      const float anew = fmaf(r.dt, v + r.b_out[tid], arow[tid]);
      arow[tid] = anew;
      sa_vec[tid] = anew;
    }
    __syncthreads();
  } else if (r.do_head) {
    if (tid < r.A) sa_vec[tid] = r.a[static_cast<size_t>(m) * r.A + tid];
    __syncthreads();
  }

  // ---- step head: x = a . w_in^T + b_in
  if (r.do_head) {
    ss = 0.f;
    for (int c = tid; c < n4; c += kRowThreads) {
      float xv[4];
      if ((r.A & 7) == 0) {
        // the four rows' weights as 16-byte loads, all issued before the FMA chains
        // (blocks past A re-read block 0 and are dropped)
        uint4 wv[4][kMaxA / 8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4* wrow = reinterpret_cast<const uint4*>(r.w_in + static_cast<size_t>(c * 4 + i) * r.A);
#pragma unroll
          for (int j = 0; j < kMaxA / 8; ++j) wv[i][j] = wrow[j < r.A / 8 ? j : 0];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float acc = 0.f;
#pragma unroll
          for (int j = 0; j < kMaxA / 8; ++j) {
            if (j < r.A / 8) {
              const __nv_bfloat16* w8 = reinterpret_cast<const __nv_bfloat16*>(&wv[i][j]);
#pragma unroll
              for (int e = 0; e < 8; ++e) acc = fmaf(sa_vec[j * 8 + e], __bfloat162float(w8[e]), acc);
            }
          }
          xv[i] = acc + r.b_in[c * 4 + i];
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n = c * 4 + i;
          const __nv_bfloat16* wrow = r.w_in + static_cast<size_t>(n) * r.A;
          float acc = 0.f;
          for (int a = 0; a < r.A; ++a) acc = fmaf(sa_vec[a], __bfloat162float(wrow[a]), acc);
          xv[i] = acc + r.b_in[n];
        }
      }
      const float4 x = make_float4(xv[0], xv[1], xv[2], xv[3]);
      *reinterpret_cast<float4*>(xs + c * 4) = x;
      *reinterpret_cast<float4*>(xrow + c * 4) = x;
      ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
    }
  }

  // ---- the row's sum of squares for a normalising GEMM prologue
  if (r.ssq) {
    const float tot = block_sum(ss, red);
    if (tid < r.ssq_tiles) r.ssq[static_cast<size_t>(tid) * r.M + m] = tid == 0 ? tot : 0.f;
  }

  // ---- AdaRMSNorm + static-scale quantisation into the next GEMM's operand
  if (r.do_quant) {
    const float rr = rsqrtf(block_sum(ss, red) / N + r.eps);
    const float rs = rs_q;
    for (int c = tid; c < n4; c += kRowThreads) {
      const float4 x = *reinterpret_cast<const float4*>(xs + c * 4);
      const int u = (c - tid) / kRowThreads;
      const float4 sc = u == 0 ? scale_v[0] : u == 1 ? scale_v[1] : *reinterpret_cast<const float4*>(r.scale + c * 4);
      const float4 sh = u == 0 ? shift_v[0] : u == 1 ? shift_v[1] : *reinterpret_cast<const float4*>(r.shift + c * 4);
      float4 h;
      h.x = fmaf(x.x * rr, 1.f + sc.x, sh.x);
      h.y = fmaf(x.y * rr, 1.f + sc.y, sh.y);
      h.z = fmaf(x.z * rr, 1.f + sc.z, sh.z);
      h.w = fmaf(x.w * rr, 1.f + sc.w, sh.w);
      if (r.q_fp8 == kQNvfp4AsF16) {
        // a 16-element block is four consecutive threads' columns (c = tid + 256 u): their
        // amax by two shuffles; every lane of the warp takes part (N is a multiple of 128)
        float a = fmaxf(fmaxf(fabsf(h.x), fabsf(h.y)), fmaxf(fabsf(h.z), fabsf(h.w)));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        float den;
        const float bs = nvfp4_block(a, rs, &den);
        const __half2 lo = nvfp4_pair(h.x, h.y, bs, den), hi = nvfp4_pair(h.z, h.w, bs, den);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&lo);
        u.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(static_cast<__half*>(r.q) + static_cast<size_t>(m) * N + c * 4) = u;
      } else {
        store_q4(r.q, static_cast<size_t>(m) * N + c * 4, h, r.q_fp8, rs);
      }
    }
  }
  if (r.stamp_kind == 2) {   // the decision's last kernel: latest CTA end
    __syncthreads();
    if (tid == 0) atomicMax(r.stamp + 1, global_ns());
  }
  if (tl_on) {
    tt[2] = global_ns();
    tl_record(r.tl, kTlRow, 1, 0, tt);
  }
}

// ---------------------------------------------------------------- decision noise

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
// 1, 2, 3", SC'11, section 3.2): per round (hi0, lo0) = M0 * x0, (hi1, lo1) = M1 * x2,
// x <- (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0); the key is bumped by the Weyl
// constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 x, uint32_t k0, uint32_t k1) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint32_t hi0 = __umulhi(kM0, x.x), lo0 = kM0 * x.x;
    const uint32_t hi1 = __umulhi(kM1, x.z), lo1 = kM1 * x.z;
    x = make_uint4(hi1 ^ x.y ^ k0, lo1, hi0 ^ x.w ^ k1, lo0);
  }
  return x;
}

// Box-Muller (Box and Muller, 1958) on two words: u = (w + 1/2) / 2^32 in (0, 1).
__device__ __forceinline__ float2 box_muller(uint32_t wa, uint32_t wb) {
  const double ua = (static_cast<double>(wa) + 0.5) * 0x1p-32;
  const double ub = (static_cast<double>(wb) + 0.5) * 0x1p-32;
  const double rad = sqrt(-2.0 * log(ua));
  double sn, cs;
  sincospi(2.0 * ub, &sn, &cs);
  return make_float2(static_cast<float>(rad * cs), static_cast<float>(rad * sn));
}

__global__ void philox_noise_kernel(float* __restrict__ out, int64_t n, uint32_t k0, uint32_t k1, uint32_t c_lo,
                                    uint32_t c_hi, uint32_t* __restrict__ raw) {
  const int64_t b = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (b * 4 >= n) return;
  const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(b), static_cast<uint32_t>(b >> 32), c_lo, c_hi),
                                k0, k1);
  if (raw) reinterpret_cast<uint4*>(raw)[b] = w;
  const float2 z01 = box_muller(w.x, w.y), z23 = box_muller(w.z, w.w);
  const float z[4] = {z01.x, z01.y, z23.x, z23.y};
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (b * 4 + j < n) out[b * 4 + j] = z[j];
}

// ---------------------------------------------------------------- create-time kernels

// cond[k][i]: the given vector, or the sinusoidal embedding of t_k = 1 - k/S
// ([sin(2 pi t / p_i), cos(2 pi t / p_i)], p_i geometric from 4e-3 to 4), in double;
// row S (rows = S + 1) is the embedding of the warm start's t = warm_t.
__global__ void cond_embed_kernel(double* conds, int S, int rows, int d, const float* given, float warm_t) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * d) return;
  if (given) {
    conds[idx] = static_cast<double>(given[idx]);
    return;
  }
  const int k = idx / d, i = idx % d, half = d / 2;
  const int f = i < half ? i : i - half;
  const double t = k < S ? 1.0 - static_cast<double>(k) / S : static_cast<double>(warm_t);
  const double period = 4e-3 * pow(4.0 / 4e-3, static_cast<double>(f) / (half - 1));
  const double arg = 2.0 * 3.14159265358979323846 * t / period;
  conds[idx] = i < half ? sin(arg) : cos(arg);
}

// out[k * step_stride + j] = fp32(sum_i cond[k][i] * w[j][i] + b[j]); one warp per output j.
__global__ void modtable_kernel(const double* __restrict__ conds, int S, int d, const __nv_bfloat16* __restrict__ w,
                                const float* __restrict__ b, int nout, float* __restrict__ out, size_t step_stride) {
  const int j = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (j >= nout) return;
  const __nv_bfloat16* wr = w + static_cast<size_t>(j) * d;
  for (int k = 0; k < S; ++k) {
    const double* c = conds + static_cast<size_t>(k) * d;
    double acc = 0.0;
    for (int i = lane; i < d; i += 32) acc += c[i] * static_cast<double>(__bfloat162float(wr[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) out[k * step_stride + j] = static_cast<float>(acc + static_cast<double>(b[j]));
  }
}

__global__ void warm_mix_kernel(float* __restrict__ a, const float* __restrict__ prev, const float* __restrict__ noise,
                                int M, int A, int e, float tau) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= M * A) return;
  const int m = idx / A, j = idx % A;
  const int src = min(m + e, M - 1);
  a[idx] = fmaf(tau, noise[idx], (1.0f - tau) * prev[src * A + j]);
}

__global__ void quant_e4m3_kernel(const float* __restrict__ x, int64_t n, float scale, uint8_t* __restrict__ codes) {
  const float rs = 1.0f / scale;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    codes[i] = e4m3(x[i] * rs);
}

}  // namespace

namespace {

// y[m][n] = bf16(sum_j planes[j][m][n] * fp32(sa * sw)), slices summed in order j = 0..s-1;
// with vt, columns n >= nv0 also go to vt[(n - nv0) * m_pad + m].
__global__ void __launch_bounds__(256) qkv_finalize_kernel(const float* __restrict__ planes, int s, size_t n4,
                                                           const float* __restrict__ sa,
                                                           const float* __restrict__ sw, __nv_bfloat16* out,
                                                           __nv_bfloat16* vt, int N, int nv0, int m_pad) {
  pdl_trigger();
  const float ds = __fmul_rn(*sa, *sw);
  pdl_wait();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float4 acc = reinterpret_cast<const float4*>(planes)[i];
    for (int j = 1; j < s; ++j) {
      const float4 v = reinterpret_cast<const float4*>(planes + static_cast<size_t>(j) * n4 * 4)[i];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * ds, acc.y * ds);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * ds, acc.w * ds);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    reinterpret_cast<uint2*>(out)[i] = u;
    const int n = static_cast<int>((i * 4) % static_cast<size_t>(N));
    if (vt && n >= nv0) {   // N and nv0 are multiples of 4: the quad lies in the V columns
      const size_t m = (i * 4) / static_cast<size_t>(N);
      __nv_bfloat16* col = vt + static_cast<size_t>(n - nv0) * m_pad + m;
      col[0] = __low2bfloat16(lo);
      col[m_pad] = __high2bfloat16(lo);
      col[2 * static_cast<size_t>(m_pad)] = __low2bfloat16(hi);
      col[3 * static_cast<size_t>(m_pad)] = __high2bfloat16(hi);
    }
  }
}

}  // namespace

cudaError_t qkv_finalize_launch(const float* planes, int s, int M, int N, const float* sa, const float* sw,
                                __nv_bfloat16* out, __nv_bfloat16* vt, int nv0, int m_pad, const LaunchOpts& o) {
  if (N % 4 || (vt && (nv0 % 4 || nv0 < 0 || nv0 > N || m_pad < M))) return cudaErrorInvalidValue;
  const size_t n4 = static_cast<size_t>(M) * N / 4;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((n4 + 255) / 256, 1216));
  return launch(qkv_finalize_kernel, dim3(blocks), dim3(256), 0, o, planes, s, n4, sa, sw, out, vt, N, nv0, m_pad);
}

cudaError_t row_launch(const RowArgs& r, const LaunchOpts& o) {
  const size_t smem = static_cast<size_t>(r.N) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = allow_max_dynamic_smem(reinterpret_cast<const void*>(row_kernel));
    if (e != cudaSuccess) return e;
  }
  RowArgs ra = r;
  ra.tl = o.tl;
  return launch(row_kernel, dim3(static_cast<unsigned>(r.M)), dim3(kRowThreads), smem, o, ra);
}

cudaError_t philox_noise_launch(float* out, int64_t n, uint64_t seed, uint64_t counter, uint32_t* raw,
                                cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = (n + 3) / 4;
  philox_noise_kernel<<<static_cast<unsigned>((blocks + 127) / 128), 128, 0, st>>>(
      out, n, static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32), static_cast<uint32_t>(counter),
      static_cast<uint32_t>(counter >> 32), raw);
  return cudaGetLastError();
}

cudaError_t cond_embed_launch(double* conds, int S, int d, const float* given, float warm_t, cudaStream_t st) {
  const int rows = S + (warm_t > 0.f ? 1 : 0);
  const int n = rows * d;
  cond_embed_kernel<<<(n + 255) / 256, 256, 0, st>>>(conds, S, rows, d, given, warm_t);
  return cudaGetLastError();
}

cudaError_t warm_mix_launch(float* a, const float* prev, const float* noise, int M, int A, int e, float tau,
                            cudaStream_t st) {
  const int n = M * A;
  warm_mix_kernel<<<(n + 255) / 256, 256, 0, st>>>(a, prev, noise, M, A, e, tau);
  return cudaGetLastError();
}

cudaError_t modtable_launch(const double* conds, int S, int d, const __nv_bfloat16* w_mod, const float* b_mod,
                            int nout, float* out, size_t out_step_stride, cudaStream_t st) {
  const int warps = 8;
  modtable_kernel<<<(nout + warps - 1) / warps, warps * 32, 0, st>>>(conds, S, d, w_mod, b_mod, nout, out,
                                                                     out_step_stride);
  return cudaGetLastError();
}

cudaError_t quant_e4m3_launch(const float* x, int64_t n, float scale, uint8_t* codes, cudaStream_t st) {
  quant_e4m3_kernel<<<1184, 256, 0, st>>>(x, n, scale, codes);
  return cudaGetLastError();
}

}  // namespace fm
