// O-projection GEMM with the attention branch's consumer fused into its epilogue.
//
// The consumer of the O GEMM (blog post "Embodied inference acceleration", section
// "Static quantisation": gated residual + AdaRMSNorm + static FP8 convert, emitting the
// next GEMM's operand) needs whole rows of the product: the RMS of x runs over every
// column. The separate K-split GEMM leaves that to a row kernel (one more kernel and one
// more programmatic-dependent-launch hand-off). Here one thread-block cluster spans all
// N / 128 column tiles of the O projection (N = d <= 1024: at most 8 CTAs) and each CTA
// takes the whole K range of its 128 weight rows, so every CTA finishes its columns of
// x <- x + gate * (A W^T) * fp32(s_a * s_w) in its own epilogue; the per-row sums of
// squares of the new x are exchanged across the cluster (st.async into each peer's
// shared memory, counted on its mbarrier) and summed in fixed rank order, and each CTA
// normalises, modulates and quantises its own columns:
//   q2 = E4M3(x / sqrt(mean(x^2) + eps) * (1 + scale) + shift) * (1 / s_q)).
// The MMA is the skinny GEMM's swap-AB tcgen05 kind::f8f6f4 (weight rows = MMA M = 128,
// activation rows = MMA N = M rounded up to 16); all K blocks of the weights are copied
// in before the programmatic-dependent-launch wait, the activations after it.

#include <cuda_fp8.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace fm {

namespace {

constexpr int kThreads = 256;      // 8 warps: two per TMEM lane quarter in the epilogue
constexpr int kTile = 128;         // weight rows (output columns) per CTA
constexpr int kBlk = 128;          // K bytes per block
constexpr int kWBlk = kTile * kBlk;   // 16 KB of packed weights per K block
constexpr int kMaxStages = 8;
constexpr int kMaxRows = 64;       // activation rows (MMA N) this kernel serves
constexpr int kMaxCluster = 8;

struct OcParams {
  const uint8_t* wpk;   // packed, pre-swizzled weight tiles [N/128][K/128][128][128 B] (E4M3)
  int M, N, nkb, n_pad, chunk;
  const float* sa;      // static scale of the attention output (the activation operand)
  const float* sw;      // weight scale
  const float* gate;    // [N] gate of the attention branch
  float* x;             // [M][N] residual stream, in/out
  const float* scale;   // [N] pre-MLP modulation
  const float* shift;
  const float* sq;      // static scale of q2
  float eps;
  uint8_t* q;           // [M][N] E4M3 codes (the gate|up GEMM's operand)
  int* err;
  // diagnostic timeline (nullptr = off): entry, after the PDL wait, MMAs complete,
  // row statistics received, outputs written, exit
  unsigned long long* tl;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct OcSmem {
  size_t w, a, ssq, part, rr, bar, total;
};
__host__ __device__ inline OcSmem oc_smem(int nkb, int n_pad) {
  OcSmem s;
  s.w = 0;
  s.a = static_cast<size_t>(nkb) * kWBlk;
  s.ssq = s.a + static_cast<size_t>(nkb) * n_pad * kBlk;               // [cluster][kMaxRows] fp32
  s.part = s.ssq + static_cast<size_t>(kMaxCluster) * kMaxRows * 4;   // [4 quarters][kMaxRows]
  s.rr = s.part + static_cast<size_t>(4) * kMaxRows * 4;              // [kMaxRows]
  s.bar = align_up(s.rr + kMaxRows * 4, 64);
  s.total = s.bar + (kMaxStages + 2) * 8 + 16;
  return s;
}

__global__ void __launch_bounds__(kThreads) o_consumer_kernel(const __grid_constant__ CUtensorMap tmA,
                                                              const OcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(smem_raw), 1024));
  __shared__ int s_abort;
  const OcSmem sp = oc_smem(p.nkb, p.n_pad);
  uint8_t* w_tiles = smem + sp.w;
  uint8_t* a_tiles = smem + sp.a;
  float* s_ssq = reinterpret_cast<float*>(smem + sp.ssq);     // [rank][m] received sums of squares
  float* s_part = reinterpret_cast<float*>(smem + sp.part);   // [quarter][m]
  float* s_rr = reinterpret_cast<float*>(smem + sp.rr);       // [m] 1 / RMS
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + sp.bar);
  uint64_t* done = full + kMaxStages;
  uint64_t* ssq_bar = done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ssq_bar + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int nt = blockIdx.x;
  const int csize = static_cast<int>(gridDim.x);   // the cluster spans every column tile
  const int nst = p.nkb / p.chunk;
  const uint32_t a_blk_bytes = static_cast<uint32_t>(p.n_pad) * kBlk;
  const uint32_t ncols = p.n_pad <= 32 ? 32u : 64u;
  const bool tl_on = p.tl != nullptr && tid == 0;
  __shared__ uint64_t tt[kTlStamps];
  if (tl_on)
    for (int i = 0; i < kTlStamps; ++i) tt[i] = 0;
  if (tl_on) tt[0] = global_ns();

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < nst; ++i) mbar_init(&full[i], 1);
    mbar_init(done, 1);
    mbar_init(ssq_bar, 1);
    fence_mbar_init();
    // every cluster rank sends one sum of squares per (padded) row
    mbar_arrive_expect_tx(ssq_bar, static_cast<uint32_t>(csize * p.n_pad * 4));
    tma_prefetch_desc(&tmA);
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tmem_slot, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive_relaxed();   // paired with the wait before the first remote store
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();   // after TMEM is held (see the skinny GEMM)

  // per-create constants of this thread's output column, fetched before the wait
  const int quarter = warp & 3, colset = warp >> 2;
  const int n_local = quarter * 32 + lane;   // TMEM lane == weight row == output column
  const int col = nt * kTile + n_local;
  const float g = p.gate[col];
  const float sc = 1.f + p.scale[col];
  const float sh = p.shift[col];
  const float ds = __fmul_rn(*p.sa, *p.sw);
  const float rs = 1.0f / *p.sq;

  if (tid == 0) {
    // ---------------- producer: every weight K block before the wait, the activations after
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_a = l2_policy_evict_last();
    const uint8_t* wsrc = p.wpk + static_cast<size_t>(nt) * p.nkb * kWBlk;
    const uint32_t w_stage = static_cast<uint32_t>(p.chunk) * kWBlk;
    for (int i = 0; i < nst; ++i) {
      mbar_arrive_expect_tx(&full[i], w_stage + p.chunk * a_blk_bytes);
      bulk_load(w_tiles + static_cast<size_t>(i) * w_stage, wsrc + static_cast<size_t>(i) * w_stage, w_stage, &full[i],
                pol_w);
    }
    pdl_wait();   // the attention output is written by the previous kernel
    if (tl_on) tt[1] = global_ns();
    for (int i = 0; i < nst; ++i)
      tma_load_3d(a_tiles + static_cast<size_t>(i) * p.chunk * a_blk_bytes, &tmA, &full[i], 0, 0, i * p.chunk, pol_a);
  } else if (tid == 32) {
    // ---------------- MMA issuer: all K blocks accumulate into one TMEM tile
    const uint32_t idesc = make_idesc(true, kTile, static_cast<uint32_t>(p.n_pad));
    for (int st = 0; st < nst; ++st) {
      if (!mbar_wait(&full[st], 0)) {
        atomicOr(p.err, kErrPipelineTimeout);
        s_abort = 1;
        break;
      }
      tc_fence_after();
      for (int c = 0; c < p.chunk; ++c) {
        const int kb = st * p.chunk + c;
        const uint32_t wa = smem_u32(w_tiles + static_cast<size_t>(kb) * kWBlk);
        const uint32_t aa = smem_u32(a_tiles + static_cast<size_t>(kb) * a_blk_bytes);
#pragma unroll
        for (int k = 0; k < kBlk / 32; ++k)
          tc_mma<true>(tmem, sw128_kmajor_desc(wa + k * 32), sw128_kmajor_desc(aa + k * 32), idesc,
                       (kb > 0 || k > 0) ? 1u : 0u);
      }
    }
    tc_commit(done);
  }

  // ---------------- epilogue: the gated residual of this CTA's columns for every row
  pdl_wait();   // x was written by an earlier kernel
  if (!mbar_wait(done, 0)) {
    atomicOr(p.err, kErrPipelineTimeout);
    s_abort = 1;
  }
  if (tl_on) tt[2] = global_ns();
  tc_fence_after();
  __syncthreads();
  const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  // warps w and w + 4 share lane quarter w % 4 and take alternate 16-row chunks (at most
  // two each: n_pad <= 64)
  float xv[2][16];
  __syncwarp();   // tcgen05.ld is warp-collective
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = colset * 16 + h * 32;
    if (c >= p.n_pad) break;
    float v[16];
    tmem_ld16(t_row + static_cast<uint32_t>(c), v);
    float xo[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)   // every row's old x first: the loads in flight together
      xo[i] = c + i < p.M ? p.x[static_cast<size_t>(c + i) * p.N + col] : 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      xv[h][i] = c + i < p.M ? fmaf(g, v[i] * ds, xo[i]) : 0.f;
      float s2 = xv[h][i] * xv[h][i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
      if (lane == 0) s_part[quarter * kMaxRows + c + i] = s2;
    }
  }
  __syncthreads();
  // this CTA's share of each row's sum of squares, pushed to every rank (slot = own rank)
  cluster_wait();   // every peer has started: its shared memory exists
  if (tid < p.n_pad) {
    const float s = ((s_part[tid] + s_part[kMaxRows + tid]) + s_part[2 * kMaxRows + tid]) + s_part[3 * kMaxRows + tid];
    const uint32_t rank = cluster_rank();
    const uint32_t off = smem_u32(s_ssq + rank * kMaxRows + tid);
    const uint32_t mb = smem_u32(ssq_bar);
    for (int r = 0; r < csize; ++r)
      st_async_f32(map_dsmem(off, static_cast<uint32_t>(r)), s, map_dsmem(mb, static_cast<uint32_t>(r)));
  }
  if (!mbar_wait(ssq_bar, 0)) {
    atomicOr(p.err, kErrPipelineTimeout);
    s_abort = 1;
  }
  if (tl_on) tt[3] = global_ns();
  // every rank's sums have arrived; the relaxed arrive, waited before exit, keeps this
  // CTA alive while its peers may still be storing into it
  cluster_arrive_relaxed();
  if (tid < p.M) {
    float t = 0.f;
    for (int r = 0; r < csize; ++r) t += s_ssq[r * kMaxRows + tid];   // fixed rank order
    s_rr[tid] = rsqrtf(t / static_cast<float>(p.N) + p.eps);
  }
  __syncthreads();
  if (s_abort == 0) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = colset * 16 + h * 32;
      if (c >= p.n_pad) break;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int m = c + i;
        if (m < p.M) {
          const float hv = fmaf(xv[h][i] * s_rr[m], sc, sh);
          const size_t idx = static_cast<size_t>(m) * p.N + col;
          p.x[idx] = xv[h][i];
          p.q[idx] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(hv * rs, __NV_SATFINITE, __NV_E4M3));
        }
      }
    }
  }
  if (tl_on) tt[4] = global_ns();
  // on an abandoned pipeline, let copies already in flight land before the CTA exits
  if (s_abort != 0 && tid == 0)
    for (int i = 0; i < nst; ++i) mbar_wait(&full[i], 0, 100000000ull);
  cluster_wait();
  tc_fence_before();
  __syncthreads();
  if (tl_on) {
    tt[5] = global_ns();
    tl_record(p.tl, kTlGemm, 1, 0, tt);
  }
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

}  // namespace

int o_consumer_plan(int M, int N, int K, OConsumerShape* g) {
  if (M < 1 || M > kMaxRows || N % kTile || N / kTile < 1 || N / kTile > kMaxCluster || K % kBlk ||
      K / kBlk < 1 || K / kBlk > kMaxStages * 4)
    return FM_ERR_SHAPE;
  g->M = M;
  g->N = N;
  g->K = K;
  g->n_pad = (M + 15) / 16 * 16;
  g->nkb = K / kBlk;
  int chunk = std::min(4, g->nkb);
  while (g->nkb % chunk) --chunk;
  g->chunk = chunk;
  if (g->nkb / chunk > kMaxStages) return FM_ERR_SHAPE;
  g->smem = 1024 + oc_smem(g->nkb, g->n_pad).total;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
      g->smem + 512 > static_cast<size_t>(optin))
    return FM_ERR_SHAPE;
  if (g->smem > 226 * 1024) return FM_ERR_SHAPE;
  return FM_OK;
}

bool o_consumer_tmap(CUtensorMap* map, const void* a, const OConsumerShape& g) {
  return make_tmap_kblocks(map, a, 1, static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.M),
                           static_cast<uint32_t>(g.n_pad), static_cast<uint32_t>(g.chunk));
}

cudaError_t o_consumer_configure() {
  return configure_once(3, [] { return allow_max_dynamic_smem(reinterpret_cast<const void*>(o_consumer_kernel)); });
}

cudaError_t o_consumer_launch(const CUtensorMap& tmA, const void* wpk, const OConsumerShape& g, const float* sa,
                              const float* sw, const float* gate, float* x, const float* scale, const float* shift,
                              const float* sq, float eps, uint8_t* q, int* err, const LaunchOpts& o) {
  OcParams p;
  p.wpk = static_cast<const uint8_t*>(wpk);
  p.M = g.M;
  p.N = g.N;
  p.nkb = g.nkb;
  p.n_pad = g.n_pad;
  p.chunk = g.chunk;
  p.sa = sa;
  p.sw = sw;
  p.gate = gate;
  p.x = x;
  p.scale = scale;
  p.shift = shift;
  p.sq = sq;
  p.eps = eps;
  p.q = q;
  p.err = err;
  p.tl = o.tl;
  LaunchOpts lo = o;
  const unsigned tiles = static_cast<unsigned>(g.N / kTile);
  lo.cluster = dim3(tiles, 1, 1);
  return launch(o_consumer_kernel, dim3(tiles, 1, 1), dim3(kThreads), g.smem, lo, tmA, p);
}

}  // namespace fm
