// Attention of the action chunk over [persistent prefix KV cache; the chunk's own KV].
//
// The prefix cache holds the observation- and instruction-dependent keys and
// values; it persists across decisions and is refreshed only when the
// observation changes (news article "FlashRT-PAI", section "It optimises the
// relay": reuse instruction-dependent results, refresh image-dependent ones).
// Queries, keys and values of the chunk come from the merged QKV GEMM (blog post,
// "CUDA Graph vs graph simplification": three projections sharing one input
// become one wider GEMM), whose epilogue already dequantised them to bf16.
//
// Work layout. The G = H/Hkv query heads sharing a KV head are stacked into rows
// r = h_local * M + m. A CTA owns a tile of 128 stacked rows and one contiguous
// slice of the keys; the slices of a row tile form a thread-block cluster. Both
// contractions run on tcgen05 tensor cores with bf16 operands in shared memory
// (K-major, 128-byte swizzle, the layout TMA writes) and fp32 accumulators in
// TMEM: S = Q K^T (M = 128 rows, N = slice keys, K = 128 head dims), then
// O = P V (N = 128 head dims, K = slice keys) with V held transposed. Each of the
// four warps owns 32 rows (its TMEM lane quarter), so the softmax needs no
// shuffles: pass 1 reads S for the row max and sum, the cluster exchanges them
// through distributed shared memory so every CTA normalises with the global max
// and sum, pass 2 forms P = exp(s - M) / L, rounds it to bf16 and writes the
// swizzled operand. The slices' shares of O are summed across the cluster in
// fixed slice order and quantised with the static output scale.

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace fm {

namespace {

constexpr int kThreads = 128;
constexpr int kRows = 128;           // stacked query rows per CTA (MMA M)
constexpr int kDh = 128;             // head dim
constexpr int kMaxSplit = 8;         // portable cluster size
constexpr int kMaxKc = 192;          // keys per slice (MMA N of QK^T), multiple of 64
constexpr int kTile = kRows * 128;   // bytes of one [128 rows][128 B] swizzled block
constexpr int kLdsO = kDh + 4;       // fp32 row stride of the O staging buffer
static_assert(kThreads == kDh, "one thread per head-dim row of V^T");

struct KParams {
  const __nv_bfloat16* qkv;    // [M][ldq]
  int ldq;
  const __nv_bfloat16* kpre;   // [P][Hkv][Dh] of this layer
  const __nv_bfloat16* vtpre;  // [Hkv][Dh][p_pad] of this layer (transposed)
  int p_pad;
  void* out;
  const float* s_out;
  int out_fp8;
  int M, P, H, Hkv, G, kc, nsplit;
  int* err;
};

__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a [rows][128 B] block with
// the 128-byte swizzle (the block base is 1024-byte aligned).
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 32 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  float a[16], b[16];
  tmem_ld16(taddr, a);
  tmem_ld16(taddr + 16, b);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[i] = a[i];
    v[16 + i] = b[i];
  }
}

__host__ __device__ inline size_t main_bytes(int kc) {
  // Q: 2 blocks; K: kc rows x 256 B; V^T and P: kc/64 blocks each
  return 2 * static_cast<size_t>(kTile) + static_cast<size_t>(kc) * 256 + 2 * static_cast<size_t>(kc / 64) * kTile;
}

__host__ __device__ inline size_t staging_bytes(int kc) {
  const size_t o = static_cast<size_t>(kRows) * kLdsO * 4;   // O staging aliases the operand tiles
  const size_t m = main_bytes(kc);
  return ((m > o ? m : o) + 1023) / 1024 * 1024;
}

__global__ void __launch_bounds__(kThreads) attn_kernel(const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int kc = p.kc;
  const int kblk = kc / 64;   // 64-key blocks of the slice
  uint8_t* sQ = smem;                                         // 2 blocks: dims 0-63, 64-127
  uint8_t* sK = sQ + 2 * kTile;                               // 2 blocks of [kc rows][128 B]
  uint8_t* sVt = sK + static_cast<size_t>(kc) * 256;          // kblk blocks of [128 dims][128 B]
  uint8_t* sP = sVt + static_cast<size_t>(kblk) * kTile;      // kblk blocks of [128 rows][128 B]
  float* sO = reinterpret_cast<float*>(smem);                 // [128][kLdsO] fp32 after both MMAs
  float* sML = reinterpret_cast<float*>(smem + staging_bytes(kc));   // [128][2] slice max, sum
  uint64_t* bar = reinterpret_cast<uint64_t*>(sML + kRows * 2);      // S done, O done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);
  __shared__ int s_abort;

  const int split = blockIdx.x;
  const int qt = blockIdx.y;
  const int g = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int nkeys = p.P + p.M;
  const int t0 = split * kc;
  const int nvalid = min(kc, nkeys - t0);
  const uint32_t ncols = (kc + kDh) <= 256 ? 256u : 512u;

  if (tid == 0) {
    s_abort = 0;
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tmem_slot, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();   // after TMEM is held: a later GEMM waiting on this grid cannot starve it

  const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVta = smem_u32(sVt), sPa = smem_u32(sP);

  // ---- prefix keys and transposed values of this slice (written before this graph ran)
  for (int idx = tid; idx < kc * 16; idx += kThreads) {
    const int i = idx >> 4, c16 = idx & 15;   // key row, 16-byte chunk of its 256 bytes
    const int t = t0 + i;
    const uint32_t dst = sKa + (c16 >> 3) * (kc * 128) + swz(i, c16 & 7);
    if (t < p.P)
      cp_async16(dst, p.kpre + (static_cast<size_t>(t) * p.Hkv + g) * kDh + c16 * 8);
    else if (t >= nkeys)
      st_shared_v4(dst, make_uint4(0, 0, 0, 0));
  }
  // V^T rows: thread d copies head-dim row d, 8 keys (16 bytes) at a time. The cache
  // row is padded with zeros from P to P_pad, so a group straddling the end of the
  // prefix is copied whole; its keys >= P are overwritten with the chunk's values.
  const int ngrp = kc / 8;   // 8-key groups of the slice
  {
    const int d = tid;   // kThreads == kDh
    const __nv_bfloat16* vrow = p.vtpre + (static_cast<size_t>(g) * kDh + d) * p.p_pad;
    for (int grp = 0; grp < ngrp; ++grp) {
      const int t = t0 + grp * 8;
      const uint32_t dst = sVta + (grp >> 3) * kTile + swz(d, grp & 7);
      if (t < p.P)
        cp_async16(dst, vrow + t);
      else
        st_shared_v4(dst, make_uint4(0, 0, 0, 0));
    }
  }
  cp_async_commit();
  pdl_wait();   // Q, K, V of the chunk are written by the QKV GEMM

  // ---- stacked query rows and the chunk's own keys (rows P..P+M-1 of the key axis)
  for (int idx = tid; idx < kRows * 16; idx += kThreads) {
    const int r = idx >> 4, c16 = idx & 15;
    const int R = qt * kRows + r;
    const uint32_t dst = sQa + (c16 >> 3) * kTile + swz(r, c16 & 7);
    if (R < p.G * p.M) {
      const int hl = R / p.M, m = R % p.M;
      cp_async16(dst, p.qkv + static_cast<size_t>(m) * p.ldq + (g * p.G + hl) * kDh + c16 * 8);
    } else {
      st_shared_v4(dst, make_uint4(0, 0, 0, 0));
    }
  }
  const int c_lo = max(t0, p.P), c_hi = min(t0 + kc, nkeys);
  const int nchunk = c_hi > c_lo ? c_hi - c_lo : 0;   // <= kc
  const __nv_bfloat16* vstage = reinterpret_cast<const __nv_bfloat16*>(sP);   // [nchunk][128] staging
  for (int idx = tid; idx < nchunk * 16; idx += kThreads) {
    const int t = c_lo + (idx >> 4), c16 = idx & 15;
    const __nv_bfloat16* row = p.qkv + static_cast<size_t>(t - p.P) * p.ldq;
    cp_async16(sKa + (c16 >> 3) * (kc * 128) + swz(t - t0, c16 & 7), row + (p.H + g) * kDh + c16 * 8);
    cp_async16(sPa + static_cast<uint32_t>(((t - c_lo) * kDh + c16 * 8) * 2), row + (p.H + p.Hkv + g) * kDh + c16 * 8);
  }
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();   // V^T groups and the staged chunk values are in place
  // the chunk's own values, transposed shared -> shared into V^T (keys along K)
  if (nchunk > 0) {
    const int d = tid;   // kThreads == kDh
    for (int t = c_lo; t < c_hi; ++t) {
      const int key = t - t0, grp = key >> 3;
      const uint16_t v = reinterpret_cast<const uint16_t*>(vstage)[(t - c_lo) * kDh + d];
      const uint32_t addr = sVta + (grp >> 3) * kTile + swz(d, grp & 7) + (key & 7) * 2;
      asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
    }
  }
  fence_async_smem();   // generic-proxy shared-memory writes -> tensor-core reads
  __syncthreads();

  // ---- S = Q K^T into TMEM columns [0, kc)
  if (tid == 0) {
    tc_fence_after();
    const uint32_t idesc = make_idesc(false, kRows, static_cast<uint32_t>(kc));
#pragma unroll
    for (int b = 0; b < 2; ++b) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc_mma<false>(tmem, sw128_kmajor_desc(sQa + b * kTile + k * 32),
                      sw128_kmajor_desc(sKa + b * (kc * 128) + k * 32), idesc, (b | k) ? 1u : 0u);
    }
    tc_commit(&bar[0]);
  }
  if (!mbar_wait(&bar[0], 0)) {
    atomicOr(p.err, kErrPipelineTimeout);
    s_abort = 1;
  }
  tc_fence_after();
  __syncwarp();

  const int r = warp * 32 + lane;   // this thread's row == its TMEM lane
  const uint32_t t_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const float kscale = 1.4426950408889634f * rsqrtf(static_cast<float>(kDh));   // log2(e) / sqrt(Dh)

  // ---- pass 1: row max and sum of exp over this slice
  float mrow = -INFINITY, lrow = 0.f;
  for (int c = 0; c < kc; c += 32) {
    float v[32];
    tmem_ld32(t_row + static_cast<uint32_t>(c), v);
    float mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      v[e] = c + e < nvalid ? v[e] * kscale : -INFINITY;
      mx = fmaxf(mx, v[e]);
    }
    const float mnew = fmaxf(mrow, mx);
    if (mnew == -INFINITY) continue;   // every key of this chunk lies past the slice end
    float sum = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) sum += exp2f(v[e] - mnew);
    lrow = lrow * exp2f(mrow - mnew) + sum;
    mrow = mnew;
  }
  sML[r * 2] = mrow;
  sML[r * 2 + 1] = lrow;

  // ---- exchange the slice statistics across the cluster: global max and sum per row
  cluster_sync_all();
  float gmax = -INFINITY, gsum = 0.f;
  {
    const uint32_t ml_local = smem_u32(sML + r * 2);
    float mq[kMaxSplit], lq[kMaxSplit];
#pragma unroll
    for (int q = 0; q < kMaxSplit; ++q) {
      if (q < p.nsplit) {
        const uint32_t a = map_dsmem(ml_local, static_cast<uint32_t>(q));
        mq[q] = ld_dsmem_f32(a);
        lq[q] = ld_dsmem_f32(a + 4);
      }
    }
#pragma unroll
    for (int q = 0; q < kMaxSplit; ++q)
      if (q < p.nsplit) gmax = fmaxf(gmax, mq[q]);
#pragma unroll
    for (int q = 0; q < kMaxSplit; ++q)
      if (q < p.nsplit) gsum += lq[q] * exp2f(mq[q] - gmax);
  }

  // ---- pass 2: P = bf16(exp(s - M) / L) into the swizzled A operand of P V
  const float ginv = 1.0f / gsum;
  for (int c = 0; c < kc; c += 32) {
    float v[32];
    tmem_ld32(t_row + static_cast<uint32_t>(c), v);
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = c + e < nvalid ? exp2f(v[e] * kscale - gmax) * ginv : 0.f;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {   // four 8-key chunks of 16 bytes
      const int key = c + ch * 8;
      uint4 u;
      u.x = pack_bf16(v[ch * 8 + 0], v[ch * 8 + 1]);
      u.y = pack_bf16(v[ch * 8 + 2], v[ch * 8 + 3]);
      u.z = pack_bf16(v[ch * 8 + 4], v[ch * 8 + 5]);
      u.w = pack_bf16(v[ch * 8 + 6], v[ch * 8 + 7]);
      st_shared_v4(sPa + (key >> 6) * kTile + swz(r, (key & 63) >> 3), u);
    }
  }
  tc_fence_before();
  fence_async_smem();
  __syncthreads();

  // ---- O = P V into TMEM columns [kc, kc + 128)
  if (tid == 0) {
    tc_fence_after();
    const uint32_t idesc = make_idesc(false, kRows, kDh);
    for (int b = 0; b < kblk; ++b) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc_mma<false>(tmem + static_cast<uint32_t>(kc), sw128_kmajor_desc(sPa + b * kTile + k * 32),
                      sw128_kmajor_desc(sVta + b * kTile + k * 32), idesc, (b | k) ? 1u : 0u);
    }
    tc_commit(&bar[1]);
  }
  if (!mbar_wait(&bar[1], 0)) {
    atomicOr(p.err, kErrPipelineTimeout);
    s_abort = 1;
  }
  tc_fence_after();
  __syncwarp();
  // this slice's share of O (already normalised by the global sum) to shared memory
  for (int c = 0; c < kDh; c += 32) {
    float v[32];
    tmem_ld32(t_row + static_cast<uint32_t>(kc + c), v);
#pragma unroll
    for (int e = 0; e < 32; e += 4)
      *reinterpret_cast<float4*>(sO + r * kLdsO + c + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
  }

  // ---- sum the slices' shares across the cluster in fixed slice order, quantise.
  // A thread owns 4 adjacent head-dim columns of one row (32 threads per row, 4 rows
  // in flight per CTA) and issues the loads of all slices before summing.
  cluster_sync_all();
  if (s_abort == 0) {
    const int rank = static_cast<int>(cluster_rank());
    const int rows_per = (kRows + p.nsplit - 1) / p.nsplit;
    const int e4 = lane * 4;
    const float rs = p.out_fp8 ? 1.0f / *p.s_out : 1.0f;
    const uint32_t o_local = smem_u32(sO);
    uint32_t peer[kMaxSplit];
#pragma unroll
    for (int q = 0; q < kMaxSplit; ++q) peer[q] = q < p.nsplit ? map_dsmem(o_local, static_cast<uint32_t>(q)) : 0u;
    const int r_end = min(kRows, (rank + 1) * rows_per);
    for (int rr = rank * rows_per + warp; rr < r_end; rr += kThreads / 32) {
      const int R = qt * kRows + rr;
      if (R >= p.G * p.M) break;
      const uint32_t off = static_cast<uint32_t>((rr * kLdsO + e4) * 4);
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
        uchar4 cc;
        cc.x = static_cast<uint8_t>(__nv_cvt_float_to_fp8(acc.x * rs, __NV_SATFINITE, __NV_E4M3));
        cc.y = static_cast<uint8_t>(__nv_cvt_float_to_fp8(acc.y * rs, __NV_SATFINITE, __NV_E4M3));
        cc.z = static_cast<uint8_t>(__nv_cvt_float_to_fp8(acc.z * rs, __NV_SATFINITE, __NV_E4M3));
        cc.w = static_cast<uint8_t>(__nv_cvt_float_to_fp8(acc.w * rs, __NV_SATFINITE, __NV_E4M3));
        *reinterpret_cast<uchar4*>(static_cast<uint8_t*>(p.out) + oidx) = cc;
      } else {
        uint2 u;
        u.x = pack_bf16(acc.x, acc.y);
        u.y = pack_bf16(acc.z, acc.w);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + oidx) = u;
      }
    }
  }
  cluster_sync_all();   // peers may still be reading this CTA's share
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// v [L][rows][Hkv][Dh] -> vt[l][g][d][tok_begin + t] with row stride p_pad.
__global__ void transpose_v_kernel(const __nv_bfloat16* __restrict__ v, __nv_bfloat16* __restrict__ vt, int L,
                                   int rows, int Hkv, int p_pad, int tok_begin) {
  const size_t total = static_cast<size_t>(L) * rows * Hkv * kDh;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int d = static_cast<int>(i % kDh);
    size_t rest = i / kDh;
    const int g = static_cast<int>(rest % Hkv);
    rest /= Hkv;
    const int t = static_cast<int>(rest % rows);
    const int l = static_cast<int>(rest / rows);
    vt[((static_cast<size_t>(l) * Hkv + g) * kDh + d) * p_pad + tok_begin + t] = v[i];
  }
}

}  // namespace

int attn_plan(int M, int P, int* kc, int* nsplit) {
  const int keys = P + M;
  int ns = (keys + 63) / 64;
  if (ns > kMaxSplit) ns = kMaxSplit;
  int per = (keys + ns - 1) / ns;
  per = (per + 63) / 64 * 64;
  if (per > kMaxKc) return FM_ERR_SHAPE;
  *kc = per;
  *nsplit = (keys + per - 1) / per;
  return FM_OK;
}

size_t attn_smem_bytes(int kc) { return 1024 + staging_bytes(kc) + kRows * 2 * 4 + 64; }

cudaError_t attn_configure() { return allow_max_dynamic_smem(reinterpret_cast<const void*>(attn_kernel)); }

cudaError_t attn_launch(const AttnArgs& a, const LaunchOpts& o) {
  KParams p;
  p.qkv = a.qkv;
  p.ldq = (a.H + 2 * a.Hkv) * kDh;
  p.kpre = a.kpre;
  p.vtpre = a.vtpre;
  p.p_pad = a.p_pad;
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
  p.err = a.err;
  const int rows = p.G * p.M;
  const dim3 grid(static_cast<unsigned>(a.nsplit), static_cast<unsigned>((rows + kRows - 1) / kRows),
                  static_cast<unsigned>(a.Hkv));
  LaunchOpts lo = o;
  lo.cluster = dim3(static_cast<unsigned>(a.nsplit), 1, 1);
  return launch(attn_kernel, grid, dim3(kThreads), attn_smem_bytes(a.kc), lo, p);
}

cudaError_t transpose_v_launch(const __nv_bfloat16* v, __nv_bfloat16* vt, int L, int rows, int Hkv, int p_pad,
                               int tok_begin, cudaStream_t st) {
  transpose_v_kernel<<<1184, 256, 0, st>>>(v, vt, L, rows, Hkv, p_pad, tok_begin);
  return cudaGetLastError();
}

}  // namespace fm
