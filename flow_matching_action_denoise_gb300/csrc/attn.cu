// Attention of the action chunk over [persistent prefix KV cache; the chunk's own KV].
//
// The prefix cache holds the observation- and instruction-dependent keys and
// values; it persists across decisions and is refreshed only when the
// observation changes (news article "FlashRT-PAI", section "It optimises the
// relay": reuse instruction-dependent results, refresh image-dependent ones).
// Queries, keys and values of the chunk come from the merged QKV GEMM (blog post,
// "CUDA Graph vs graph simplification": three projections sharing one input
// become one wider GEMM), whose epilogue already dequantised them and rounded
// them to bf16, so this kernel only copies rows into shared memory.
//
// Layout of the work: the G = H/Hkv query heads that share a KV head are stacked
// into rows r = h_local * M + m, so one K/V tile serves all of them. A CTA owns
// 64 stacked rows (4 warps x 16) and one contiguous slice of the keys; the
// slices of one row tile form a thread-block cluster. Each warp runs QK^T and PV
// on bf16 tensor cores (m16n8k16, fp32 accumulate). The softmax statistics (row
// max and sum) are exchanged across the cluster through distributed shared
// memory, so the probabilities are normalised before they are rounded to bf16;
// the slices' shares of O are summed across the cluster in fixed slice order and
// quantised with the static output scale.

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace fm {

namespace {

constexpr int kThreads = 128;
constexpr int kRows = 64;        // stacked query rows per CTA
constexpr int kDh = 128;         // head dim
constexpr int kLds = kDh + 8;    // bf16 elements per shared row (272 B: conflict-free ldmatrix)
constexpr int kChunk = 64;       // keys per online-softmax chunk
constexpr int kMaxSplit = 8;     // portable cluster size

struct KParams {
  const __nv_bfloat16* qkv;   // [M][ldq]
  int ldq;
  const __nv_bfloat16* kpre;
  const __nv_bfloat16* vpre;
  void* out;
  const float* s_out;
  int out_fp8;
  int M, P, H, Hkv, G, kc, nsplit;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* dst, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(dst) = u;
}

__global__ void __launch_bounds__(kThreads) attn_kernel(const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* sK = sQ + kRows * kLds;
  __nv_bfloat16* sV = sK + p.kc * kLds;
  float* sML = reinterpret_cast<float*>(sV + p.kc * kLds);   // [64][2]: slice max (log2 units), slice sum
  float* sStat = sML + kRows * 2;                             // [64][2]: global max, global sum
  float* sO = reinterpret_cast<float*>(sK);                   // [64][128] fp32, aliases K/V after compute

  const int split = blockIdx.x;
  const int qt = blockIdx.y;
  const int g = blockIdx.z;
  const int tid = threadIdx.x;
  const int nkeys = p.P + p.M;
  const int t0 = split * p.kc;
  const int nvalid = min(p.kc, nkeys - t0);

  pdl_trigger();

  // ---- prefix keys/values of this slice (written before this graph ran): 16-byte
  // asynchronous copies, all in flight together; rows past the last key are zeroed.
  for (int idx = tid; idx < p.kc * 16; idx += kThreads) {
    const int i = idx >> 4, c = idx & 15;
    const int t = t0 + i;
    if (t < p.P) {
      const size_t off = (static_cast<size_t>(t) * p.Hkv + g) * kDh + c * 8;
      cp_async16(sK + i * kLds + c * 8, p.kpre + off);
      cp_async16(sV + i * kLds + c * 8, p.vpre + off);
    } else if (t >= nkeys) {
      *reinterpret_cast<uint4*>(sK + i * kLds + c * 8) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sV + i * kLds + c * 8) = make_uint4(0, 0, 0, 0);
    }
  }
  pdl_wait();   // Q, K, V of the chunk are written by the QKV GEMM

  // ---- stacked query rows and the chunk's own keys/values (key rows P..P+M-1):
  // bf16 rows of the QKV GEMM's dequantised output, copied asynchronously.
  for (int idx = tid; idx < kRows * 16; idx += kThreads) {
    const int r = idx >> 4, c = idx & 15;
    const int R = qt * kRows + r;
    if (R < p.G * p.M) {
      const int hl = R / p.M, m = R % p.M;
      cp_async16(sQ + r * kLds + c * 8, p.qkv + static_cast<size_t>(m) * p.ldq + (g * p.G + hl) * kDh + c * 8);
    } else {
      *reinterpret_cast<uint4*>(sQ + r * kLds + c * 8) = make_uint4(0, 0, 0, 0);
    }
  }
  const int c_lo = max(t0, p.P), c_hi = min(t0 + p.kc, nkeys);
  for (int idx = tid; idx < (c_hi > c_lo ? (c_hi - c_lo) : 0) * 16; idx += kThreads) {
    const int t = c_lo + (idx >> 4), c = idx & 15;
    const __nv_bfloat16* row = p.qkv + static_cast<size_t>(t - p.P) * p.ldq;
    cp_async16(sK + (t - t0) * kLds + c * 8, row + (p.H + g) * kDh + c * 8);
    cp_async16(sV + (t - t0) * kLds + c * 8, row + (p.H + p.Hkv + g) * kDh + c * 8);
  }
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();

  // ---- per-warp attention over this slice, two passes over the keys:
  // pass 1 finds the row max and the row sum of exp over the slice; the cluster
  // exchanges them so every CTA holds the global max M and sum L of each row;
  // pass 2 forms the normalised probabilities P = exp(s - M) / L, rounds them to
  // bf16 for the tensor-core PV product, and accumulates this slice's share of O.
  // The rounding points are thus those of softmax-then-bf16, independent of how
  // the keys are split across CTAs.
  const int warp = tid >> 5, lane = tid & 31;
  const int r0 = warp * 16;
  uint32_t qf[8][4];
  {
    const uint32_t qbase = smem_u32(sQ + (r0 + (lane & 15)) * kLds + (lane >> 4) * 8);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) ldsm_x4(qbase + ks * 32, qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
  }
  const float kscale = 1.4426950408889634f * rsqrtf(static_cast<float>(kDh));   // log2(e) / sqrt(Dh)
  const int nchunks = (nvalid + kChunk - 1) / kChunk;
  const int mat = lane >> 3;

  // S = Q K^T for one 64-key chunk, scaled to log2 units, masked past nvalid.
  auto scores = [&](int ch, float (&s)[8][4]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      const int key = ch * kChunk + np * 16 + (lane & 7) + (mat >> 1) * 8;
      const uint32_t kbase = smem_u32(sK + key * kLds + (mat & 1) * 8);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + ks * 32, b0, b1, b2, b3);
        mma_bf16(s[2 * np], qf[ks], b0, b1);
        mma_bf16(s[2 * np + 1], qf[ks], b2, b3);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = ch * kChunk + nt * 8 + (lane & 3) * 2 + (e & 1);
        s[nt][e] = key < nvalid ? s[nt][e] * kscale : -INFINITY;
      }
    }
  };

  // ---- pass 1: row max and sum of exp over this slice
  float mrow[2] = {-INFINITY, -INFINITY};
  float lrow[2] = {0.f, 0.f};
  for (int ch = 0; ch < nchunks; ++ch) {
    float s[8][4];
    scores(ch, s);
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) mx[e >> 1] = fmaxf(mx[e >> 1], s[nt][e]);
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
      const float mnew = fmaxf(mrow[hr], mx[hr]);
      lrow[hr] *= exp2f(mrow[hr] - mnew);
      mrow[hr] = mnew;
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) lrow[e >> 1] += exp2f(s[nt][e] - mrow[e >> 1]);
    }
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 1);
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 2);
  }
  {
    const int rlo = r0 + (lane >> 2), rhi = rlo + 8;
    if ((lane & 3) == 0) {
      sML[rlo * 2] = mrow[0];
      sML[rlo * 2 + 1] = lrow[0];
      sML[rhi * 2] = mrow[1];
      sML[rhi * 2 + 1] = lrow[1];
    }
  }
  // ---- exchange the slice statistics across the cluster: global max and sum per row
  cluster_sync_all();
  if (tid < kRows) {
    const uint32_t ml_local = smem_u32(sML + tid * 2);
    float mq[kMaxSplit], lq[kMaxSplit];
#pragma unroll
    for (int q = 0; q < kMaxSplit; ++q) {
      if (q < p.nsplit) {
        const uint32_t a = map_dsmem(ml_local, static_cast<uint32_t>(q));
        mq[q] = ld_dsmem_f32(a);
        lq[q] = ld_dsmem_f32(a + 4);
      }
    }
    float mstar = -INFINITY;
#pragma unroll
    for (int q = 0; q < kMaxSplit; ++q)
      if (q < p.nsplit) mstar = fmaxf(mstar, mq[q]);
    float lsum = 0.f;
#pragma unroll
    for (int q = 0; q < kMaxSplit; ++q)
      if (q < p.nsplit) lsum += lq[q] * exp2f(mq[q] - mstar);
    sStat[tid * 2] = mstar;
    sStat[tid * 2 + 1] = lsum;
  }
  __syncthreads();
  const float gmax[2] = {sStat[(r0 + (lane >> 2)) * 2], sStat[(r0 + (lane >> 2) + 8) * 2]};
  const float gsum[2] = {sStat[(r0 + (lane >> 2)) * 2 + 1], sStat[(r0 + (lane >> 2) + 8) * 2 + 1]};

  // ---- pass 2: O_slice = bf16(exp(s - M) / L) V
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  for (int ch = 0; ch < nchunks; ++ch) {
    float s[8][4];
    scores(ch, s);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = exp2f(s[nt][e] - gmax[e >> 1]) / gsum[e >> 1];
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t a[4];
      a[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      a[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      a[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      a[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      const int key = ch * kChunk + kk * 16 + (lane & 7) + (mat & 1) * 8;
      const uint32_t vbase = smem_u32(sV + key * kLds + (mat >> 1) * 8);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + dp * 32, b0, b1, b2, b3);
        mma_bf16(o[2 * dp], a, b0, b1);
        mma_bf16(o[2 * dp + 1], a, b2, b3);
      }
    }
  }

  // ---- this slice's share of O into shared memory (over the K/V tiles)
  __syncthreads();
  {
    const int rlo = r0 + (lane >> 2), rhi = rlo + 8;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int col = nt * 8 + (lane & 3) * 2;
      *reinterpret_cast<float2*>(sO + rlo * kDh + col) = make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2*>(sO + rhi * kDh + col) = make_float2(o[nt][2], o[nt][3]);
    }
  }

  // ---- sum the slices' shares across the cluster in fixed slice order, quantise.
  // A thread owns 4 adjacent head-dim columns of one row (32 threads per row,
  // 4 rows in flight per CTA) and issues the loads of all slices before summing.
  cluster_sync_all();
  {
    const int rank = static_cast<int>(cluster_rank());
    const int rows_per = (kRows + p.nsplit - 1) / p.nsplit;
    const int e4 = lane * 4;
    const float rs = p.out_fp8 ? 1.0f / *p.s_out : 1.0f;
    const uint32_t o_local = smem_u32(sO);
    uint32_t peer[kMaxSplit];
#pragma unroll
    for (int q = 0; q < kMaxSplit; ++q) peer[q] = q < p.nsplit ? map_dsmem(o_local, static_cast<uint32_t>(q)) : 0u;
    const int r_end = min(kRows, (rank + 1) * rows_per);
    for (int r = rank * rows_per + warp; r < r_end; r += kThreads / 32) {
      const int R = qt * kRows + r;
      if (R >= p.G * p.M) break;
      const uint32_t off = static_cast<uint32_t>((r * kDh + e4) * 4);
      float4 v[kMaxSplit];
#pragma unroll
      for (int q = 0; q < kMaxSplit; ++q)
        if (q < p.nsplit) v[q] = ld_dsmem_f32x4(peer[q] + off);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < kMaxSplit; ++q) {
        if (q < p.nsplit) {
          acc.x += v[q].x;
          acc.y += v[q].y;
          acc.z += v[q].z;
          acc.w += v[q].w;
        }
      }
      const int hl = R / p.M, m = R % p.M;
      const size_t oidx = static_cast<size_t>(m) * (p.H * kDh) + (g * p.G + hl) * kDh + e4;
      if (p.out_fp8) {
        uchar4 c;
        c.x = static_cast<uint8_t>(__nv_cvt_float_to_fp8(acc.x * rs, __NV_SATFINITE, __NV_E4M3));
        c.y = static_cast<uint8_t>(__nv_cvt_float_to_fp8(acc.y * rs, __NV_SATFINITE, __NV_E4M3));
        c.z = static_cast<uint8_t>(__nv_cvt_float_to_fp8(acc.z * rs, __NV_SATFINITE, __NV_E4M3));
        c.w = static_cast<uint8_t>(__nv_cvt_float_to_fp8(acc.w * rs, __NV_SATFINITE, __NV_E4M3));
        *reinterpret_cast<uchar4*>(static_cast<uint8_t*>(p.out) + oidx) = c;
      } else {
        store_bf16x4(static_cast<__nv_bfloat16*>(p.out) + oidx, acc);
      }
    }
  }
  cluster_sync_all();   // peers may still be reading this CTA's share
}

}  // namespace

void attn_plan(int M, int P, int* kc, int* nsplit) {
  const int keys = P + M;
  int ns = (keys + kChunk - 1) / kChunk;
  if (ns > kMaxSplit) ns = kMaxSplit;
  int per = (keys + ns - 1) / ns;
  per = (per + kChunk - 1) / kChunk * kChunk;
  *kc = per;
  *nsplit = (keys + per - 1) / per;
}

size_t attn_smem_bytes(int kc) {
  return 128 + static_cast<size_t>(kRows) * kLds * 2 + 2 * static_cast<size_t>(kc) * kLds * 2 + 2 * kRows * 2 * 4;
}

cudaError_t attn_configure() { return allow_max_dynamic_smem(reinterpret_cast<const void*>(attn_kernel)); }

cudaError_t attn_launch(const AttnArgs& a, const LaunchOpts& o) {
  KParams p;
  p.qkv = a.qkv;
  p.ldq = (a.H + 2 * a.Hkv) * kDh;
  p.kpre = a.kpre;
  p.vpre = a.vpre;
  p.out = a.out;
  p.s_out = a.s_out;
  p.out_fp8 = a.out_fp8;
  p.M = a.M;
  p.P = a.P;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.G = a.H / a.Hkv;
  p.kc = a.kc;
  p.nsplit = a.nsplit;
  const int rows = p.G * p.M;
  const dim3 grid(static_cast<unsigned>(a.nsplit), static_cast<unsigned>((rows + kRows - 1) / kRows),
                  static_cast<unsigned>(a.Hkv));
  LaunchOpts lo = o;
  lo.cluster = dim3(static_cast<unsigned>(a.nsplit), 1, 1);
  return launch(attn_kernel, grid, dim3(kThreads), attn_smem_bytes(a.kc), lo, p);
}

}  // namespace fm
