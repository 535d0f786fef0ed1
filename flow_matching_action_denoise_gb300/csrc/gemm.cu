// Skinny GEMM with K-split on tcgen05 tensor cores, and weight packing.
//
// Computes partial[j][m][n] = sum_{k in slice j} A[m][k] * W[n][k] for an action
// chunk of M <= 256 rows (blog post "Embodied inference acceleration", section
// "Small-M GEMM": C = sum_j A_j W_j over s K slices, FP32 partial sums reduced
// before the consumer's own transform).
//
// GB300 mapping ("swap-AB"): the weight tile is the MMA's A operand (M = 128 rows
// of W, i.e. 128 output columns n), the activations are the MMA's B operand
// (N = M rounded up to 16), so the tiny row count costs nothing in tensor-core
// shape. Each TMA transaction and each barrier round trip costs a fixed ~0.1-0.3 us
// on this part while the bytes of one transaction are nearly free up to tens of KB,
// so a pipeline stage moves `chunk` K blocks at once: the weights - the only large
// operand, packed pre-swizzled so a plain bulk copy lands them in the MMA layout -
// in one copy of chunk x 16 KB, the activations in one 3-D box of chunk K blocks.
// One elected thread issues the TMA loads, another issues tcgen05.mma into a
// TMEM accumulator; eight warps (two per TMEM lane quarter) read it back. CTAs
// (n-tile, slice j) of consecutive slices form a thread-block cluster of size cs
// that sums its partials in fixed slice order through distributed shared memory,
// so only s/cs partial planes go to global memory (deterministic, no atomics).
// Weight loads are issued before the programmatic-dependent-launch wait: they do
// not depend on the previous kernel, so they overlap its tail.

#include <cudaTypedefs.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace fm {

namespace {

constexpr int kThreads = 256;   // 8 warps: two per TMEM lane quarter in the epilogue
constexpr int kTileN = 128;                      // weight rows per CTA (MMA M)
constexpr int kBlockBytes = 128;                 // K bytes per pipeline block (one swizzle row)
constexpr int kMaxStages = 8;
constexpr int kWTileBytes = kTileN * kBlockBytes;   // 16 KB
constexpr size_t kStageCap = 196 * 1024;         // shared-memory budget for the ring
constexpr size_t kCtrlBytes = 256;

struct KParams {
  const uint8_t* wpk;       // packed, pre-swizzled weight tiles [N/128][K blocks][128][128 B]
  float* out;               // fp32 partial planes [s/cs][M][N], or
  __nv_bfloat16* out_bf16;  // when non-null (cs == s): bf16(sum * fp32(sa * sw)) [M][N]
  void* out_geglu;          // when non-null (cs == s, gate|up interleaved): Q(gelu(g) u) [M][N/2]
  uint8_t* out_qkv8;        // when non-null (cs == s): E4M3 codes of Q | K | V [M][N] with scales s_qkv[0..2]
  const float* s_qkv;
  int nq, nk;
  int geglu_fp8;
  const float* sq;          // static scale of the GeGLU output
  const float* sa;
  const float* sw;
  int M, N;
  int nkb_total, nkb_cta;
  int n_pad, stages, cs, chunk;
  const uint8_t* pf;   // a range to prefetch into L2 (each CTA its share), or nullptr
  size_t pf_bytes;
  int* err;
  // kMode 1 (residual epilogue; cs == s): x[m][n] += gate[n] * (sum * fp32(sa * sw)) for the
  // rows and columns this CTA finalises, and ssq[nt][m] = the tile's sum of x_new^2.
  // kMode 2 (normalising prologue): the activation operand of the CTA's K range is built
  // here from x: q = Q(x * rsqrt(sum_t ssq[t][m] / K + eps) * (1 + scale) + shift).
  float* x;
  const float* gate;
  float* ssq;
  const float* scale;
  const float* shift;
  const float* sqa;   // static scale of q (FP8 operands)
  float eps;
  void* q_out;        // kMode 2: n-tile 0 also stores its K range of q here
  // diagnostic timeline (nullptr = off): entry, activations requested (after the PDL
  // wait), MMAs complete, partial rows pushed, split-K rows received, outputs written, exit
  unsigned long long* tl;
};

__host__ __device__ inline uint32_t pow2_at_least(uint32_t v, uint32_t lo) {
  uint32_t p = lo;
  while (p < v) p <<= 1;
  return p;
}

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// kTm: weight rows per CTA, the MMA's M: 128, or 64 (the first or second half of a packed
// 128-row tile; plain placement only), which halves the partial bytes each CTA of a
// K-split cluster pushes to its peers. With M = 64 the accumulator's row r sits in TMEM
// lane 32 (r / 16) + r % 16: lanes 0-15 of each warp's lane quarter.
// This CTA's share of the L2 prefetch range (16-byte units; a grid-wide split).
__device__ __forceinline__ void l2_prefetch_share(const KParams& p) {
  if (!p.pf) return;
  const size_t nct = static_cast<size_t>(gridDim.x) * gridDim.y;
  const size_t cta = static_cast<size_t>(blockIdx.y) * gridDim.x + blockIdx.x;
  const size_t share = ((p.pf_bytes / 16 + nct - 1) / nct) * 16;
  const size_t lo = cta * share, hi = lo + share < p.pf_bytes ? lo + share : p.pf_bytes;
  for (size_t a = lo; a < hi; a += 65536)
    l2_prefetch_bulk(p.pf + a, static_cast<uint32_t>(hi - a < 65536 ? hi - a : 65536));
}

// Output rows are finalised in four-row groups: cluster rank o owns the groups
// g = o (mod cs) of the M rows (as its local group g / cs), so a lane's four
// consecutive accumulator columns (activation rows 4g..4g+3 of its weight row) go to
// one owner in one 16-byte store, and consecutive groups to different owners. The
// receive buffer is [slot][owned group][weight row][4 rows]: the 32 lanes of a warp
// (consecutive weight rows, one group) fill 512 contiguous bytes of one owner.
__host__ __device__ inline int owner_groups(int M, int cs) { return ((M + 3) / 4 + cs - 1) / cs; }

template <bool kFp8, int kCs, int kMode, int kTm = kTileN>
__global__ void __launch_bounds__(kThreads) skinny_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                                                               const KParams p) {
  static_assert(kTm == kTileN || (kTm == kTileN / 2 && kMode == 0), "64-row tiles: plain placement only");
  constexpr uint32_t kTmBytes = kTm * kBlockBytes;   // one K block of this CTA's weight rows
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(smem_raw), 1024));
  __shared__ int s_abort;
  __shared__ int s_issued;
  // placement with the consumer inside (kMode 1): per owned row, the sums of squares of
  // the tile's four 32-row slabs (at most 256 rows per rank)
  __shared__ float s_ssq[kMode == 1 ? 4 : 1][kMode == 1 ? 256 : 1];

  const int stages = p.stages;
  const int chunk = p.chunk;
  const uint32_t a_tile_bytes = static_cast<uint32_t>(p.n_pad) * kBlockBytes;
  const uint32_t w_stage_bytes = static_cast<uint32_t>(chunk) * kTmBytes;
  const uint32_t a_stage_bytes = static_cast<uint32_t>(chunk) * a_tile_bytes;
  uint8_t* w_tiles = smem;
  uint8_t* a_tiles = smem + static_cast<size_t>(stages) * w_stage_bytes;
  const size_t main_bytes = static_cast<size_t>(stages) * (w_stage_bytes + a_stage_bytes);
  const int groups = (p.M + 3) / 4;              // four-row groups holding a real row
  const int g_per = owner_groups(p.M, kCs);      // groups each cluster rank finalises
  float* recv = reinterpret_cast<float*>(smem + align_up(main_bytes, 1024));   // [kCs][g_per][kTm][4]
  uint8_t* ctrl = reinterpret_cast<uint8_t*>(recv) +
                  align_up(static_cast<size_t>(kCs) * g_per * kTm * 4 * sizeof(float), 1024);
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + kMaxStages;
  uint64_t* done = empty + kMaxStages;
  uint64_t* recvd = done + 1;   // the partial rows this CTA finalises have arrived from every rank
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nt = blockIdx.x;
  const int j = blockIdx.y;
  const uint32_t ncols = pow2_at_least(static_cast<uint32_t>(p.n_pad), 32);
  const bool tl_on = p.tl != nullptr && threadIdx.x == 0;
  __shared__ uint64_t tt[kTlStamps];   // timeline stamps (thread 0)
  if (tl_on)
    for (int i = 0; i < kTlStamps; ++i) tt[i] = 0;
  if (tl_on) tt[0] = global_ns();

  if (threadIdx.x == 0) {
    s_abort = 0;
    s_issued = 0;
    for (int i = 0; i < stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(done, 1);
    mbar_init(recvd, 1);
    fence_mbar_init();
    if (kCs > 1) {   // every rank sends each of its kTm weight rows' 16 bytes of every owned group
      const int rk = static_cast<int>(cluster_rank());
      const int owned = rk < groups ? (groups - 1 - rk) / kCs + 1 : 0;
      mbar_arrive_expect_tx(recvd, static_cast<uint32_t>(kCs * owned * kTm * 16));
    }
    if (kMode != 2) tma_prefetch_desc(&tmA);
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tmem_slot, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (kCs > 1) cluster_arrive_relaxed();   // paired with the wait before the first remote store
  const uint32_t tmem = *tmem_slot;
  const float ds = (p.out_bf16 || p.out_geglu || p.out_qkv8 || kMode == 1) ? __fmul_rn(*p.sa, *p.sw) : 1.0f;
  float rs_qkv[3] = {1.0f, 1.0f, 1.0f};
  if (p.out_qkv8)
    for (int i = 0; i < 3; ++i) rs_qkv[i] = 1.0f / p.s_qkv[i];
  const float rs_geglu = (p.out_geglu && p.geglu_fp8) ? 1.0f / *p.sq : 1.0f;
  // Dependents may start only once this CTA holds its TMEM: a later GEMM's CTAs that
  // wait for this grid must never be able to take the columns this CTA still needs.
  pdl_trigger();

  const int kb0 = j * p.nkb_cta;
  const int nst = p.nkb_cta / chunk;   // pipeline stages to run (chunk divides nkb_cta)

  if (kMode == 2 && threadIdx.x == 0) {
    // ---------------- producer: only the weights (the whole K range fits in the stages);
    // the activation operand is built by all threads below
    const uint64_t pol_w = l2_policy_evict_first();
    const uint8_t* wsrc = p.wpk + (static_cast<size_t>(nt) * p.nkb_total + kb0) * kWTileBytes;
    for (int i = 0; i < nst; ++i) {
      mbar_arrive_expect_tx(&full[i], w_stage_bytes);
      bulk_load(w_tiles + static_cast<size_t>(i) * w_stage_bytes, wsrc + static_cast<size_t>(i) * w_stage_bytes,
                w_stage_bytes, &full[i], pol_w);
    }
    l2_prefetch_share(p);   // after this CTA's own weights
    s_issued = nst;
  } else if (kMode != 2 && threadIdx.x == 0) {
    // ---------------- producer: per stage one bulk copy of chunk weight tiles (contiguous
    // in the packed layout) and one 3-D box of chunk activation K blocks
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_a = l2_policy_evict_last();
    // packed tiles are 128 rows: a 64-row CTA takes half nt % 2 of tile nt / 2, one
    // 8 KB copy per K block (the halves of consecutive blocks are 16 KB apart)
    const int tile = kTm == kTileN ? nt : nt / 2;
    const uint8_t* wsrc = p.wpk + (static_cast<size_t>(tile) * p.nkb_total + kb0) * kWTileBytes +
                          (kTm == kTileN ? 0 : static_cast<size_t>(nt % 2) * kTmBytes);
    auto load_w = [&](int slot, int st) {
      if constexpr (kTm == kTileN) {
        bulk_load(w_tiles + static_cast<size_t>(slot) * w_stage_bytes, wsrc + static_cast<size_t>(st) * w_stage_bytes,
                  w_stage_bytes, &full[slot], pol_w);
      } else {
        for (int c = 0; c < chunk; ++c)
          bulk_load(w_tiles + static_cast<size_t>(slot) * w_stage_bytes + c * kTmBytes,
                    wsrc + static_cast<size_t>(st * chunk + c) * kWTileBytes, kTmBytes, &full[slot], pol_w);
      }
    };
    const uint32_t tx = w_stage_bytes + a_stage_bytes;
    const int pre = min(stages, nst);
    for (int i = 0; i < pre; ++i) {
      mbar_arrive_expect_tx(&full[i], tx);
      load_w(i, i);
    }
    l2_prefetch_share(p);   // after this CTA's own weights
    pdl_wait();   // activations are written by the previous kernel
    if (tl_on) tt[1] = global_ns();
    for (int i = 0; i < pre; ++i)
      tma_load_3d(a_tiles + static_cast<size_t>(i) * a_stage_bytes, &tmA, &full[i], 0, 0, kb0 + i * chunk, pol_a);
    int issued = pre;
    for (int st = stages; st < nst; ++st) {
      const int slot = st % stages;
      const uint32_t use = static_cast<uint32_t>(st / stages);
      if (!mbar_wait(&empty[slot], (use - 1) & 1)) {
        atomicOr(p.err, kErrPipelineTimeout);
        s_abort = 1;
        break;
      }
      mbar_arrive_expect_tx(&full[slot], tx);
      load_w(slot, st);
      tma_load_3d(a_tiles + static_cast<size_t>(slot) * a_stage_bytes, &tmA, &full[slot], 0, 0, kb0 + st * chunk,
                  pol_a);
      ++issued;
    }
    s_issued = issued;
  }
  if constexpr (kMode == 2) {
    // ---------------- normalising prologue: AdaRMSNorm + static quantise of x into the
    // swizzled K-major operand tiles of this CTA's K range (blog post, section "Static
    // quantisation": the input-dependent RMS is computed at run time, gamma folded into W).
    // Thread t owns 16-byte chunk t % nchunk of every row (t / nchunk + i * rstep).
    constexpr int kEb = kFp8 ? 1 : 2;
    constexpr int kPerChunk = 16 / kEb;   // elements per 16-byte chunk
    const int K = p.nkb_total * (kBlockBytes / kEb);
    const int k_lo = kb0 * (kBlockBytes / kEb);
    const int nchunk = p.nkb_cta * (kBlockBytes / 16);
    const int ci = static_cast<int>(threadIdx.x) % nchunk;
    const int rstep = kThreads / nchunk;
    const int k0 = k_lo + ci * kPerChunk;
    float sc[kPerChunk], sh[kPerChunk];   // per-create constants: fetched before the wait
#pragma unroll
    for (int e = 0; e < kPerChunk; e += 4) {
      const float4 a = *reinterpret_cast<const float4*>(p.scale + k0 + e);
      const float4 b = *reinterpret_cast<const float4*>(p.shift + k0 + e);
      sc[e] = 1.f + a.x; sc[e + 1] = 1.f + a.y; sc[e + 2] = 1.f + a.z; sc[e + 3] = 1.f + a.w;
      sh[e] = b.x; sh[e + 1] = b.y; sh[e + 2] = b.z; sh[e + 3] = b.w;
    }
    const float rs = kFp8 ? 1.0f / *p.sqa : 1.0f;
    __shared__ float s_rr[256];
    pdl_wait();   // x and its tile sums are written by the previous kernel
    if (tl_on) tt[1] = global_ns();
    if (static_cast<int>(threadIdx.x) < p.M) {
      const int ntile = K / kTileN;
      float ss = 0.f;
      int t = 0;
      for (; t + 4 <= ntile; t += 4) {   // independent loads in flight together
        const float a = p.ssq[t * p.M + threadIdx.x], b = p.ssq[(t + 1) * p.M + threadIdx.x];
        const float c = p.ssq[(t + 2) * p.M + threadIdx.x], d = p.ssq[(t + 3) * p.M + threadIdx.x];
        ss += a;
        ss += b;
        ss += c;
        ss += d;
      }
      for (; t < ntile; ++t) ss += p.ssq[t * p.M + threadIdx.x];
      s_rr[threadIdx.x] = rsqrtf(ss / static_cast<float>(K) + p.eps);
    }
    __syncthreads();
    const int kbl = ci / (kBlockBytes / 16), c16 = ci % (kBlockBytes / 16);   // K block within the range, chunk
    uint8_t* tile = a_tiles + static_cast<size_t>(kbl / chunk) * a_stage_bytes + (kbl % chunk) * a_tile_bytes;
    // rows in batches of kBatch, their x loads issued together (the loads are the latency)
    constexpr int kBatch = kFp8 ? 4 : 8;
    for (int m0 = static_cast<int>(threadIdx.x) / nchunk; m0 < p.n_pad; m0 += kBatch * rstep) {
      float4 xv[kBatch][kPerChunk / 4];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int m = m0 + b * rstep;
        const float* xr = p.x + static_cast<size_t>(m < p.M ? m : 0) * K + k0;
#pragma unroll
        for (int e = 0; e < kPerChunk / 4; ++e)
          xv[b][e] = m < p.M ? *reinterpret_cast<const float4*>(xr + 4 * e) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int m = m0 + b * rstep;
        if (m >= p.n_pad) break;
        uint4 u = make_uint4(0, 0, 0, 0);
        if (m < p.M) {
          const float rr = s_rr[m];
          float h[kPerChunk];
#pragma unroll
          for (int e = 0; e < kPerChunk / 4; ++e) {
            h[4 * e] = fmaf(xv[b][e].x * rr, sc[4 * e], sh[4 * e]);
            h[4 * e + 1] = fmaf(xv[b][e].y * rr, sc[4 * e + 1], sh[4 * e + 1]);
            h[4 * e + 2] = fmaf(xv[b][e].z * rr, sc[4 * e + 2], sh[4 * e + 2]);
            h[4 * e + 3] = fmaf(xv[b][e].w * rr, sc[4 * e + 3], sh[4 * e + 3]);
          }
          uint32_t* w = &u.x;
          if constexpr (kFp8) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              w[q] = static_cast<uint32_t>(__nv_cvt_float_to_fp8(h[4 * q] * rs, __NV_SATFINITE, __NV_E4M3)) |
                     (static_cast<uint32_t>(__nv_cvt_float_to_fp8(h[4 * q + 1] * rs, __NV_SATFINITE, __NV_E4M3)) << 8) |
                     (static_cast<uint32_t>(__nv_cvt_float_to_fp8(h[4 * q + 2] * rs, __NV_SATFINITE, __NV_E4M3)) << 16) |
                     (static_cast<uint32_t>(__nv_cvt_float_to_fp8(h[4 * q + 3] * rs, __NV_SATFINITE, __NV_E4M3)) << 24);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(h[2 * q], h[2 * q + 1]);
              w[q] = *reinterpret_cast<const uint32_t*>(&b2);
            }
          }
          if (nt == 0 && p.q_out)
            *reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.q_out) + (static_cast<size_t>(m) * K + k0) * kEb) = u;
        }
        st_shared_v4(smem_u32(tile) + static_cast<uint32_t>(m * 128 + ((c16 ^ (m & 7)) << 4)), u);
      }
    }
    fence_async_smem();   // generic-proxy writes -> tensor-core reads
    __syncthreads();
  }
  if (threadIdx.x == 32) {
    // ---------------- MMA issuer
    const uint32_t idesc = make_idesc(kFp8, kTm, static_cast<uint32_t>(p.n_pad));
    for (int st = 0; st < nst; ++st) {
      const int slot = st % stages;
      const uint32_t use = static_cast<uint32_t>(st / stages);
      if (!mbar_wait(&full[slot], use & 1)) {
        atomicOr(p.err, kErrPipelineTimeout);
        s_abort = 1;
        break;
      }
      tc_fence_after();
      for (int c = 0; c < chunk; ++c) {
        const uint32_t wa = smem_u32(w_tiles + static_cast<size_t>(slot) * w_stage_bytes + c * kTmBytes);
        const uint32_t aa = smem_u32(a_tiles + static_cast<size_t>(slot) * a_stage_bytes + c * a_tile_bytes);
#pragma unroll
        for (int k = 0; k < kBlockBytes / 32; ++k)
          tc_mma<kFp8>(tmem, sw128_kmajor_desc(wa + k * 32), sw128_kmajor_desc(aa + k * 32), idesc,
                       (st > 0 || c > 0 || k > 0) ? 1u : 0u);
      }
      tc_commit(&empty[slot]);
    }
    tc_commit(done);
  }

  // ---------------- epilogue. Each CTA pushes its fp32 partials into the owners'
  // receive buffers (slot = its own rank): a lane holds one weight row's accumulator
  // columns, i.e. consecutive activation rows, so each group of four goes out as one
  // 16-byte remote shared-memory store counted on the owner's mbarrier. Each owner
  // then sums its groups over the cs slots in slice order, turns each 4 x 4 block
  // (four weight rows of four activation rows) around by lane shuffles and writes
  // its rows with 16-byte stores. With cs == 1 the push is a local store.
  pdl_wait();
  if (!mbar_wait(done, 0)) {
    atomicOr(p.err, kErrPipelineTimeout);
    s_abort = 1;
  }
  if (tl_on) tt[2] = global_ns();
  tc_fence_after();
  __syncthreads();
  const bool abort = s_abort != 0;
  // warps w and w + 4 share TMEM lane quarter w % 4 and take alternate 16-column chunks
  const int quarter = warp & 3, colset = warp >> 2;
  // TMEM lane == weight row within the tile (64-row tiles: lanes 0-15 of each quarter)
  const int n_local = kTm == kTileN ? quarter * 32 + lane : quarter * 16 + (lane & 15);
  const bool lane_has_row = kTm == kTileN || lane < 16;
  const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  const int rank = kCs > 1 ? static_cast<int>(cluster_rank()) : 0;
  const uint32_t recv_base = smem_u32(recv);
  if (kCs > 1) cluster_wait();   // every peer has started: its receive buffer exists
  __syncwarp();                  // tcgen05.ld is warp-collective
  const uint32_t recvd_addr = smem_u32(recvd);
  for (int c = colset * 16; c < p.n_pad; c += 32) {
    float v[16];
    tmem_ld16(t_row + static_cast<uint32_t>(c), v);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int g = (c >> 2) + b;   // activation rows 4g..4g+3 (rows past M hold zeros)
      if (g < groups && lane_has_row) {
        const int o = g % kCs, lg = g / kCs;   // owner rank and its local group
        const uint32_t addr = recv_base + static_cast<uint32_t>((((rank * g_per + lg) * kTm) + n_local) * 16);
        if (kCs > 1)   // counted on the owner's mbarrier
          st_async_v4(map_dsmem(addr, static_cast<uint32_t>(o)), v[4 * b], v[4 * b + 1], v[4 * b + 2],
                      v[4 * b + 3], map_dsmem(recvd_addr, static_cast<uint32_t>(o)));
        else
          st_shared_v4(addr, make_uint4(__float_as_uint(v[4 * b]), __float_as_uint(v[4 * b + 1]),
                                        __float_as_uint(v[4 * b + 2]), __float_as_uint(v[4 * b + 3])));
      }
    }
  }
  if (tl_on) tt[3] = global_ns();
  if (kCs > 1) {
    // every rank's partial rows for this CTA have landed (no cluster-wide release barrier);
    // the relaxed arrive, waited before exit, keeps this CTA alive while peers store into it
    if (!mbar_wait(recvd, 0)) atomicOr(p.err, kErrPipelineTimeout);
    cluster_arrive_relaxed();
  } else {
    __syncthreads();
  }
  if (tl_on) tt[4] = global_ns();
  if (!abort) {
    const int part = j / kCs;
    const int owned = rank < groups ? (groups - 1 - rank) / kCs + 1 : 0;
    const bool residual = kMode == 1 && !p.out_geglu && !p.out_qkv8 && !p.out_bf16;
    // thread <-> (weight row n of the tile, owned group lg); kTm * owned is a multiple of
    // 64, so every warp runs the same number of trips (the shuffles need all lanes)
    for (int idx = threadIdx.x; idx < kTm * owned; idx += kThreads) {
      const int n = idx % kTm, lg = idx / kTm;
      const float* src = recv + (lg * kTm + n) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < kCs; ++q) {   // slices in order
        const float4 v = *reinterpret_cast<const float4*>(src + q * g_per * kTm * 4);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      // lanes 4k..4k+3 hold weight rows n0..n0+3 of the same four activation rows; after
      // the transpose lane t4 holds activation row 4g + t4, columns n0..n0+3
      const int t4 = n & 3;
      transpose4x4(acc.x, acc.y, acc.z, acc.w, t4);
      const int m = 4 * (lg * kCs + rank) + t4;
      const int c4 = n - t4;
      const size_t col = static_cast<size_t>(nt) * kTm + c4;
      if constexpr (kMode == 1) {
        if (residual) {
          // gated residual on the finished sum, and this warp's share of the row's sum
          // of squares (lanes t4, t4 + 4, ..., t4 + 28: its 32 weight rows)
          float ssq = 0.f;
          if (m < p.M) {
            const float4 g = *reinterpret_cast<const float4*>(p.gate + col);
            float4* xp = reinterpret_cast<float4*>(p.x + static_cast<size_t>(m) * p.N + col);
            float4 xv = *xp;
            xv.x = fmaf(g.x, acc.x * ds, xv.x);
            xv.y = fmaf(g.y, acc.y * ds, xv.y);
            xv.z = fmaf(g.z, acc.z * ds, xv.z);
            xv.w = fmaf(g.w, acc.w * ds, xv.w);
            *xp = xv;
            ssq = xv.x * xv.x + xv.y * xv.y + xv.z * xv.z + xv.w * xv.w;
          }
          ssq += __shfl_xor_sync(0xffffffffu, ssq, 4);
          ssq += __shfl_xor_sync(0xffffffffu, ssq, 8);
          ssq += __shfl_xor_sync(0xffffffffu, ssq, 16);
          if (lane < 4) s_ssq[n >> 5][4 * lg + t4] = ssq;
          continue;
        }
      }
      if (m >= p.M) continue;
      if (p.out_geglu) {
        // the four columns are (gate, up) of GeGLU columns 2L and 2L+1 of this tile's 64:
        // m = gelu_tanh(g) * u, quantised
        float mv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float x = (e ? acc.z : acc.x) * ds;
          const float u = (e ? acc.w : acc.y) * ds;
          mv[e] = 0.5f * x * (1.f + tanhf(0.7978845608028654f * fmaf(0.044715f * x, x * x, x))) * u;
        }
        const size_t fidx = static_cast<size_t>(m) * (p.N / 2) + static_cast<size_t>(nt) * (kTm / 2) + c4 / 2;
        if (p.geglu_fp8) {
          uchar2 c;
          c.x = static_cast<uint8_t>(__nv_cvt_float_to_fp8(mv[0] * rs_geglu, __NV_SATFINITE, __NV_E4M3));
          c.y = static_cast<uint8_t>(__nv_cvt_float_to_fp8(mv[1] * rs_geglu, __NV_SATFINITE, __NV_E4M3));
          *reinterpret_cast<uchar2*>(static_cast<uint8_t*>(p.out_geglu) + fidx) = c;
        } else {
          const __nv_bfloat162 b = __floats2bfloat162_rn(mv[0], mv[1]);
          *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.out_geglu) + fidx) = b;
        }
      } else if (p.out_qkv8) {
        // the 4 columns share a section (sections are multiples of 128 columns)
        const int c0 = static_cast<int>(col);
        const float rs = c0 < p.nq ? rs_qkv[0] : (c0 < p.nq + p.nk ? rs_qkv[1] : rs_qkv[2]);
        uchar4 cq;
        cq.x = static_cast<uint8_t>(__nv_cvt_float_to_fp8((acc.x * ds) * rs, __NV_SATFINITE, __NV_E4M3));
        cq.y = static_cast<uint8_t>(__nv_cvt_float_to_fp8((acc.y * ds) * rs, __NV_SATFINITE, __NV_E4M3));
        cq.z = static_cast<uint8_t>(__nv_cvt_float_to_fp8((acc.z * ds) * rs, __NV_SATFINITE, __NV_E4M3));
        cq.w = static_cast<uint8_t>(__nv_cvt_float_to_fp8((acc.w * ds) * rs, __NV_SATFINITE, __NV_E4M3));
        *reinterpret_cast<uchar4*>(p.out_qkv8 + static_cast<size_t>(m) * p.N + col) = cq;
      } else if (p.out_bf16) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * ds, acc.y * ds);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * ds, acc.w * ds);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&lo);
        u.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(p.out_bf16 + static_cast<size_t>(m) * p.N + col) = u;
      } else {
        *reinterpret_cast<float4*>(p.out + (static_cast<size_t>(part) * p.M + m) * p.N + col) = acc;
      }
    }
    if constexpr (kMode == 1) {
      if (residual) {   // the row's sum of squares over the tile: its four 32-row slabs in order
        __syncthreads();
        for (int lr = threadIdx.x; lr < 4 * owned; lr += kThreads) {
          const int m = 4 * ((lr >> 2) * kCs + rank) + (lr & 3);
          if (m < p.M)
            p.ssq[static_cast<size_t>(nt) * p.M + m] = ((s_ssq[0][lr] + s_ssq[1][lr]) + s_ssq[2][lr]) + s_ssq[3][lr];
        }
      }
    }
  }

  if (tl_on) tt[5] = global_ns();
  // On an abandoned pipeline, let copies already in flight land before the CTA exits.
  if (abort && threadIdx.x == 0) {
    const int issued = s_issued;
    for (int slot = 0; slot < stages && slot < issued; ++slot) {
      const uint32_t last_use = static_cast<uint32_t>((issued - 1 - slot) / stages);
      mbar_wait(&full[slot], last_use & 1, 100000000ull);
    }
  }
  if (kCs > 1) cluster_wait();
  tc_fence_before();
  __syncthreads();
  if (tl_on) {
    tt[6] = global_ns();
    tl_record(p.tl, kTlGemm, gridDim.y, blockIdx.y, tt);
  }
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// ---------------------------------------------------------------- packing kernels

__global__ void amax_fold_kernel(const float* __restrict__ w, const float* __restrict__ gamma, int N, int K,
                                 unsigned* __restrict__ amax) {
  const size_t total = static_cast<size_t>(N) * K;
  float m = 0.f;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float g = gamma ? gamma[i % K] : 1.0f;
    m = fmaxf(m, fabsf(__fmul_rn(w[i], g)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax, __float_as_uint(m));   // non-negative floats order as uints
}

__global__ void scale_from_amax_kernel(const unsigned* __restrict__ amax, float* __restrict__ scale) {
  const float a = __uint_as_float(*amax);
  *scale = a > 0.f ? a / 448.0f : 1.0f;
}

__global__ void set_one_kernel(float* p) { *p = 1.0f; }

// FP8: one thread writes 16 bytes (16 codes) of a [128][128]-byte tile.
// Packed row n of a gate|up weight with interleave: tile t = n / 128 holds, for GeGLU
// columns j = 64t .. 64t+63, gate row j at tile row 2(j - 64t) and the matching up row
// F + j at tile row 2(j - 64t) + 1 (F = N/2), so one output tile carries both halves of
// 64 GeGLU columns and each (gate, up) pair sits in adjacent accumulator columns.
__device__ __forceinline__ size_t source_row(size_t n, int N, int interleave) {
  if (!interleave) return n;
  const size_t t = n / 128, r = n % 128;
  return (r & 1 ? static_cast<size_t>(N / 2) : 0) + t * 64 + r / 2;
}

__global__ void pack_fp8_kernel(const float* __restrict__ w, const float* __restrict__ gamma, int N, int K,
                                const float* __restrict__ scale, uint8_t* __restrict__ out, int interleave) {
  const size_t chunks = static_cast<size_t>(N) * K / 16;
  const size_t c = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  if (c >= chunks) return;
  const float rs = 1.0f / *scale;
  const size_t o = c * 16;
  const int nkb = K / 128;
  const size_t tile = o / kWTileBytes;
  const int within = static_cast<int>(o % kWTileBytes);
  const int r = within / 128, cb = within % 128;
  const int ntile = static_cast<int>(tile / nkb), kb = static_cast<int>(tile % nkb);
  const size_t n = source_row(static_cast<size_t>(ntile) * 128 + r, N, interleave);
  const int k0 = kb * 128 + cb;
  // stored at the 128-byte-swizzled position of its 16-byte chunk (the MMA layout)
  const size_t dst = tile * kWTileBytes + r * 128 + (((cb >> 4) ^ (r & 7)) << 4);
  alignas(16) uint8_t codes[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float g = gamma ? gamma[k0 + i] : 1.0f;
    const float v = __fmul_rn(__fmul_rn(w[n * K + k0 + i], g), rs);
    codes[i] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
  }
  *reinterpret_cast<uint4*>(out + dst) = *reinterpret_cast<const uint4*>(codes);
}

// BF16: one thread writes 16 bytes (8 values) of a [128][64]-element tile.
__global__ void pack_bf16_kernel(const float* __restrict__ w, const float* __restrict__ gamma, int N, int K,
                                 __nv_bfloat16* __restrict__ out, int interleave) {
  const size_t chunks = static_cast<size_t>(N) * K / 8;
  const size_t c = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  if (c >= chunks) return;
  const size_t e = c * 8;   // element offset in the packed buffer
  const int nkb = K / 64;
  const size_t tile = e / (128 * 64);
  const int within = static_cast<int>(e % (128 * 64));
  const int r = within / 64, ce = within % 64;
  const int ntile = static_cast<int>(tile / nkb), kb = static_cast<int>(tile % nkb);
  const size_t n = source_row(static_cast<size_t>(ntile) * 128 + r, N, interleave);
  const int k0 = kb * 64 + ce;
  const size_t dst = tile * (128 * 64) + r * 64 + (((ce >> 3) ^ (r & 7)) << 3);   // swizzled chunk, in elements
  alignas(16) __nv_bfloat16 vals[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float g = gamma ? gamma[k0 + i] : 1.0f;
    vals[i] = __float2bfloat16_rn(__fmul_rn(w[n * K + k0 + i], g));
  }
  *reinterpret_cast<uint4*>(out + dst) = *reinterpret_cast<const uint4*>(vals);
}

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

}  // namespace

bool make_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner, uint64_t outer,
                  uint32_t box_inner, uint32_t box_outer) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  if (reinterpret_cast<uintptr_t>(base) % 16) return false;
  const CUtensorMapDataType dt = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * static_cast<cuuint64_t>(elem_bytes)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_kblocks(CUtensorMap* map, const void* base, int elem_bytes, uint64_t K, uint64_t rows,
                       uint32_t box_rows, uint32_t blocks) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  if (reinterpret_cast<uintptr_t>(base) % 16 || (K * elem_bytes) % 128) return false;
  const CUtensorMapDataType dt = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t inner = 128 / elem_bytes;
  cuuint64_t dims[3] = {inner, rows, K / inner};
  cuuint64_t strides[2] = {K * static_cast<cuuint64_t>(elem_bytes), 128};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(inner), box_rows, blocks};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int gemm_plan(int M, int N, int K, int fp8, int s, int cs, GemmShape* g, int tile) {
  if (M < 1 || M > 256 || N <= 0 || K <= 0 || N % 128 || K % 128) return FM_ERR_SHAPE;
  if (tile != kTileN && tile != kTileN / 2) return FM_ERR_SHAPE;
  const int eb = fp8 ? 1 : 2;
  const int nkb_total = K * eb / kBlockBytes;
  if (s < 1 || nkb_total % s) return FM_ERR_SHAPE;
  if (cs < 1 || cs > 8 || (cs & (cs - 1)) || s % cs) return FM_ERR_SHAPE;
  g->M = M;
  g->N = N;
  g->K = K;
  g->fp8 = fp8;
  g->s = s;
  g->cs = cs;
  g->n_pad = (M + 15) / 16 * 16;
  g->nkb_total = nkb_total;
  g->nkb_cta = nkb_total / s;
  g->tile = tile;
  const size_t block_bytes =
      static_cast<size_t>(tile) * kBlockBytes + static_cast<size_t>(g->n_pad) * kBlockBytes;   // one K block
  const size_t recv_bytes =
      align_up(static_cast<size_t>(cs) * owner_groups(M, cs) * tile * 4 * sizeof(float), 1024);
  if (recv_bytes + block_bytes > kStageCap) return FM_ERR_SHAPE;
  // chunk: the largest divisor of nkb_cta up to 4 whose double-buffered ring fits (or a
  // single stage holding all of the CTA's K blocks)
  const size_t room = kStageCap - recv_bytes;
  int chunk = 1;
  for (int c = std::min(4, g->nkb_cta); c >= 1; --c) {
    if (g->nkb_cta % c) continue;
    const int need = std::min(2, g->nkb_cta / c);
    if (static_cast<size_t>(need) * c * block_bytes <= room) {
      chunk = c;
      break;
    }
  }
  g->chunk = chunk;
  const size_t stage_bytes = static_cast<size_t>(chunk) * block_bytes;
  int st = static_cast<int>(room / stage_bytes);
  st = std::min(st, kMaxStages);
  st = std::min(st, g->nkb_cta / chunk);
  g->stages = std::max(st, 1);
  const size_t main_bytes = g->stages * stage_bytes;
  g->smem = 1024 + align_up(main_bytes, 1024) + recv_bytes + kCtrlBytes;
  return FM_OK;
}

bool gemm_tmap_act(CUtensorMap* map, const void* a, const GemmShape& g) {
  return make_tmap_kblocks(map, a, g.fp8 ? 1 : 2, static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.M),
                           static_cast<uint32_t>(g.n_pad), static_cast<uint32_t>(g.chunk));
}

cudaError_t allow_max_dynamic_smem(const void* kernel, size_t* granted) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  const int dyn = optin - static_cast<int>(fa.sharedSizeBytes);
  if (granted) *granted = static_cast<size_t>(dyn);
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
}

cudaError_t configure_once(int family, cudaError_t (*fn)()) {
  static std::atomic<uint64_t> done[4];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (family < 0 || family >= 4 || dev >= 64) return fn();
  const uint64_t bit = 1ull << dev;
  if (done[family].load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = fn();
  if (e == cudaSuccess) done[family].fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

namespace {

template <int kMode>
cudaError_t configure_mode() {
  const void* ks[8] = {reinterpret_cast<const void*>(skinny_gemm_kernel<true, 1, kMode>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<true, 2, kMode>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<true, 4, kMode>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<true, 8, kMode>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<false, 1, kMode>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<false, 2, kMode>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<false, 4, kMode>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<false, 8, kMode>)};
  for (const void* k : ks) {
    const cudaError_t e = allow_max_dynamic_smem(k);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t configure_half_tiles() {
  const void* ks[8] = {reinterpret_cast<const void*>(skinny_gemm_kernel<true, 1, 0, kTileN / 2>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<true, 2, 0, kTileN / 2>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<true, 4, 0, kTileN / 2>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<true, 8, 0, kTileN / 2>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<false, 1, 0, kTileN / 2>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<false, 2, 0, kTileN / 2>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<false, 4, 0, kTileN / 2>),
                       reinterpret_cast<const void*>(skinny_gemm_kernel<false, 8, 0, kTileN / 2>)};
  for (const void* k : ks) {
    const cudaError_t e = allow_max_dynamic_smem(k);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t gemm_configure_impl() {
  cudaError_t e = configure_mode<0>();
  if (e == cudaSuccess) e = configure_mode<1>();
  if (e == cudaSuccess) e = configure_mode<2>();
  if (e == cudaSuccess) e = configure_half_tiles();
  return e;
}

cudaError_t launch_half_tiles(const GemmShape& g, dim3 grid, const LaunchOpts& lo, const CUtensorMap& tmA,
                              const KParams& p) {
  const dim3 blk(kThreads);
  constexpr int kH = kTileN / 2;
  switch (g.cs * 2 + (g.fp8 ? 1 : 0)) {
    case 3: return launch(skinny_gemm_kernel<true, 1, 0, kH>, grid, blk, g.smem, lo, tmA, p);
    case 5: return launch(skinny_gemm_kernel<true, 2, 0, kH>, grid, blk, g.smem, lo, tmA, p);
    case 9: return launch(skinny_gemm_kernel<true, 4, 0, kH>, grid, blk, g.smem, lo, tmA, p);
    case 17: return launch(skinny_gemm_kernel<true, 8, 0, kH>, grid, blk, g.smem, lo, tmA, p);
    case 2: return launch(skinny_gemm_kernel<false, 1, 0, kH>, grid, blk, g.smem, lo, tmA, p);
    case 4: return launch(skinny_gemm_kernel<false, 2, 0, kH>, grid, blk, g.smem, lo, tmA, p);
    case 8: return launch(skinny_gemm_kernel<false, 4, 0, kH>, grid, blk, g.smem, lo, tmA, p);
    case 16: return launch(skinny_gemm_kernel<false, 8, 0, kH>, grid, blk, g.smem, lo, tmA, p);
    default: return cudaErrorInvalidValue;
  }
}

template <int kMode>
cudaError_t launch_mode(const GemmShape& g, dim3 grid, const LaunchOpts& lo, const CUtensorMap& tmA, const KParams& p) {
  const dim3 blk(kThreads);
  switch (g.cs * 2 + (g.fp8 ? 1 : 0)) {
    case 3: return launch(skinny_gemm_kernel<true, 1, kMode>, grid, blk, g.smem, lo, tmA, p);
    case 5: return launch(skinny_gemm_kernel<true, 2, kMode>, grid, blk, g.smem, lo, tmA, p);
    case 9: return launch(skinny_gemm_kernel<true, 4, kMode>, grid, blk, g.smem, lo, tmA, p);
    case 17: return launch(skinny_gemm_kernel<true, 8, kMode>, grid, blk, g.smem, lo, tmA, p);
    case 2: return launch(skinny_gemm_kernel<false, 1, kMode>, grid, blk, g.smem, lo, tmA, p);
    case 4: return launch(skinny_gemm_kernel<false, 2, kMode>, grid, blk, g.smem, lo, tmA, p);
    case 8: return launch(skinny_gemm_kernel<false, 4, kMode>, grid, blk, g.smem, lo, tmA, p);
    case 16: return launch(skinny_gemm_kernel<false, 8, kMode>, grid, blk, g.smem, lo, tmA, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t gemm_configure() { return configure_once(0, gemm_configure_impl); }

cudaError_t gemm_launch(const void* wpk, const CUtensorMap& tmA, const GemmShape& g, float* out, int* err,
                        const LaunchOpts& o, __nv_bfloat16* out_bf16, const float* sa, const float* sw,
                        void* out_geglu, int geglu_fp8, const float* sq, uint8_t* out_qkv8, const float* s_qkv,
                        int nq, int nk, const GemmFuse* fuse, const void* l2_prefetch,
                        size_t l2_prefetch_bytes) {
  if (l2_prefetch && (reinterpret_cast<uintptr_t>(l2_prefetch) % 16 || l2_prefetch_bytes % 16))
    return cudaErrorInvalidValue;
  if ((out_bf16 || out_geglu || out_qkv8) && (g.cs != g.s || !sa || !sw)) return cudaErrorInvalidValue;
  if (out_qkv8 && (!s_qkv || nq % 128 || nk % 128)) return cudaErrorInvalidValue;
  if (out_geglu && (!sq || g.N % 128)) return cudaErrorInvalidValue;
  KParams p;
  p.wpk = static_cast<const uint8_t*>(wpk);
  p.out = out;
  p.out_bf16 = out_bf16;
  p.out_qkv8 = out_qkv8;
  p.s_qkv = s_qkv;
  p.nq = nq;
  p.nk = nk;
  p.out_geglu = out_geglu;
  p.geglu_fp8 = geglu_fp8;
  p.sq = sq;
  p.sa = sa;
  p.sw = sw;
  p.M = g.M;
  p.N = g.N;
  p.nkb_total = g.nkb_total;
  p.nkb_cta = g.nkb_cta;
  p.n_pad = g.n_pad;
  p.stages = g.stages;
  p.cs = g.cs;
  p.chunk = g.chunk;
  p.pf = static_cast<const uint8_t*>(l2_prefetch);
  p.pf_bytes = l2_prefetch ? l2_prefetch_bytes : 0;
  p.err = err;
  const int mode = fuse ? fuse->mode : 0;
  p.x = fuse ? fuse->x : nullptr;
  p.gate = fuse ? fuse->gate : nullptr;
  p.ssq = fuse ? fuse->ssq : nullptr;
  p.scale = fuse ? fuse->scale : nullptr;
  p.shift = fuse ? fuse->shift : nullptr;
  p.sqa = fuse ? fuse->sqa : nullptr;
  p.eps = fuse ? fuse->eps : 0.f;
  p.q_out = fuse ? fuse->q_out : nullptr;
  p.tl = o.tl;
  if (mode == 1 && (g.cs != g.s || !p.x || !p.gate || !p.ssq || !sa || !sw || out_bf16 || out_geglu || out_qkv8))
    return cudaErrorInvalidValue;
  if (mode == 2 && (!gemm_mode2_ok(g) || !p.x || !p.ssq || !p.scale || !p.shift || (g.fp8 && !p.sqa)))
    return cudaErrorInvalidValue;
  if (mode == 0 && !out && !out_bf16 && !out_geglu && !out_qkv8) return cudaErrorInvalidValue;
  LaunchOpts lo = o;
  lo.cluster = dim3(1, static_cast<unsigned>(g.cs), 1);
  const dim3 grid(static_cast<unsigned>(g.N / g.tile), static_cast<unsigned>(g.s), 1);
  if (g.tile != kTileN) {
    if (mode != 0) return cudaErrorInvalidValue;
    return launch_half_tiles(g, grid, lo, tmA, p);
  }
  switch (mode) {
    case 0: return launch_mode<0>(g, grid, lo, tmA, p);
    case 1: return launch_mode<1>(g, grid, lo, tmA, p);
    case 2: return launch_mode<2>(g, grid, lo, tmA, p);
    default: return cudaErrorInvalidValue;
  }
}

bool gemm_mode2_ok(const GemmShape& g) {
  const int nchunk = g.nkb_cta * (kBlockBytes / 16);
  return g.nkb_cta / g.chunk <= g.stages && nchunk <= kThreads && kThreads % nchunk == 0 && g.M <= 256;
}

size_t packed_weight_bytes(int N, int K, int fmt) {
  if (fmt == FM_FMT_FP8) return static_cast<size_t>(N) * K;
  if (fmt == FM_FMT_BF16) return static_cast<size_t>(N) * K * 2;
  if (fmt == FM_FMT_NVFP4) return nvfp4_packed_bytes(N, K);
  return 0;
}

cudaError_t weight_amax_launch(const float* w, const float* gamma, int N, int K, unsigned* amax, cudaStream_t st) {
  const cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  amax_fold_kernel<<<1184, 256, 0, st>>>(w, gamma, N, K, amax);
  return cudaGetLastError();
}

cudaError_t pack_weight(const float* w, const float* gamma, int N, int K, int fmt, void* packed, float* scale_out,
                        unsigned* amax_scratch, cudaStream_t st, int geglu_interleave) {
  const int threads = 256;
  if (fmt == FM_FMT_NVFP4) return pack_nvfp4(w, gamma, N, K, packed, scale_out, amax_scratch, st, geglu_interleave);
  if (fmt == FM_FMT_FP8) {
    cudaError_t e = weight_amax_launch(w, gamma, N, K, amax_scratch, st);
    if (e != cudaSuccess) return e;
    scale_from_amax_kernel<<<1, 1, 0, st>>>(amax_scratch, scale_out);
    const size_t chunks = static_cast<size_t>(N) * K / 16;
    pack_fp8_kernel<<<static_cast<unsigned>((chunks + threads - 1) / threads), threads, 0, st>>>(
        w, gamma, N, K, scale_out, static_cast<uint8_t*>(packed), geglu_interleave);
    return cudaGetLastError();
  }
  if (fmt == FM_FMT_BF16) {
    set_one_kernel<<<1, 1, 0, st>>>(scale_out);
    const size_t chunks = static_cast<size_t>(N) * K / 8;
    pack_bf16_kernel<<<static_cast<unsigned>((chunks + threads - 1) / threads), threads, 0, st>>>(
        w, gamma, N, K, static_cast<__nv_bfloat16*>(packed), geglu_interleave);
    return cudaGetLastError();
  }
  return cudaErrorInvalidValue;
}

}  // namespace fm
