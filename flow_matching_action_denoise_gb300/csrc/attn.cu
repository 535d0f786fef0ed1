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
// contractions run on tcgen05 tensor cores with fp32 accumulators in TMEM:
// S = Q K^T (M = 128 rows, N = slice keys, K = 128 head dims) from bf16 (or E4M3)
// operands in shared memory (K-major, 128-byte swizzle, the layout TMA writes),
// then O = P V (N = head dims of O, K = slice keys) with P read from tensor memory
// and V held transposed in shared memory. On small grids the two halves of the
// head dims of O are two CTAs that compute the same S and softmax, so each
// exchanges and sums half the O bytes (the duplicated S and exponentials run on
// otherwise idle SMs). Four warps (eight in the 256-key wide slice) share each
// TMEM lane quarter (32 rows) and split the slice's keys, so the softmax needs no
// shuffles: pass 1 reads S, takes each row part's max m_h and keeps exp(s - m_h)
// in registers with its sum; the cluster exchanges the (max, sum) pairs through
// distributed shared memory so every CTA normalises with the global max M and
// sum L; pass 2 forms P = exp(s - m_h) * exp(m_h - M) / L, rounds it to bf16 (or
// E4M3) and writes it into tensor memory. Each slice pushes its share of O
// (staged, then one bulk copy per band) into the shared memory of the CTA that
// finalises those rows, which sums the shares in fixed slice order and quantises
// with the static output scale.

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace fm {

namespace {

constexpr int kRows = 128;           // stacked query rows per CTA (MMA M)
constexpr int kDh = 128;             // head dim
constexpr int kMaxSplit = 8;         // portable cluster size
constexpr int kMaxKc = 192;          // keys per slice (MMA N of QK^T), multiple of 64, by default
constexpr int kWideKc = 256;         // the wide slice (bf16, all head dims): fewer slices per cluster
constexpr int kTile = kRows * 128;   // bytes of one [128 rows][128 B] swizzled block
// Threads of a CTA: warps split each row's keys, four (eight for the wide slice) per
// TMEM lane quarter, so that every thread keeps at most 48 scores in registers.
__host__ __device__ constexpr int attn_threads(int kc) { return kc == kWideKc ? 1024 : 512; }
static_assert(attn_threads(64) % kDh == 0 && attn_threads(kWideKc) % kDh == 0, "whole threads per head-dim row");

struct KParams {
  const __nv_bfloat16* qkv;    // [M][ldq]
  const uint8_t* qkv8;         // FP8 attention: E4M3 codes [M][ldq]
  const uint8_t* kpre8;        // FP8 attention: [P][Hkv][Dh] codes of this layer
  const uint8_t* vtpre8;       // FP8 attention: [Hkv][Dh][p16] codes (transposed)
  int p16;
  const float* s_qkv;          // FP8 attention: static scales of Q, K, V
  int ldq;
  const __nv_bfloat16* kpre;   // [P][Hkv][Dh] of this layer
  const __nv_bfloat16* vtpre;  // [Hkv][Dh][p_pad] of this layer (transposed)
  int p_pad;
  void* out;
  const float* s_out;
  int out_fp8;
  int M, P, H, Hkv, G, kc, nsplit;
  const __nv_bfloat16* vtc;    // the chunk's values transposed [Hkv][Dh][m_pad], or nullptr
  int m_pad;
  int* err;
  // diagnostic timeline (nullptr = off): entry, after the PDL wait, operands loaded, chunk
  // values transposed, S = Q K^T complete, pass 1 done, cluster peers started, statistics
  // sent, every slice's statistics received, P written, O = P V complete, O band copies
  // issued, this CTA's O band received, band summed and stored, exit
  unsigned long long* tl;
};

__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Byte offset of 16-byte chunk c (0..7) of row r inside a [rows][128 B] block with
// the 128-byte swizzle (the block base is 1024-byte aligned).
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Shared-memory plan of one CTA (byte offsets from the 1024-aligned base).
struct SmemPlan {
  size_t q, k, vt, pm, stage, recv, stats, part, bar, total;
};
// Operand tiles: Q [128 rows][Dh] (bf16: two 128-byte blocks, E4M3: one); K [kc keys][Dh]
// likewise; P in blocks of [128 rows][128 bytes] and this CTA's dv head dims of V^T in
// blocks of [dv rows][128 bytes] along the keys (bf16: kc/64 blocks of 64 keys; E4M3: the
// keys padded to a multiple of 128, one block per 128 keys).
__host__ __device__ inline int kblocks(int kc, bool fp8) { return fp8 ? (kc + 127) / 128 : kc / 64; }
// Each thread of a warp writes its TMEM lane's N (4..28, a multiple of 4) consecutive
// 32-bit columns from r, in stores of 16, 8 and 4 columns (warp-collective).
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
  static_assert(N % 4 == 0 && N >= 4 && N <= 28, "4 to 28 columns, a multiple of 4");
  constexpr int o8 = N >= 16 ? 16 : 0;
  constexpr int o4 = o8 + (N - o8 >= 8 ? 8 : 0);
  static_assert(N - o4 == 0 || N - o4 == 4, "columns left for the last store");
  if constexpr (N >= 16) {
    uint32_t a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = r[i];
    tmem_st16(taddr, a);
  }
  if constexpr (N - o8 >= 8) {
    uint32_t a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = r[o8 + i];
    tmem_st8(taddr + o8, a);
  }
  if constexpr (N - o4 == 4) {
    uint32_t a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = r[o4 + i];
    tmem_st4(taddr + o4, a);
  }
}

__host__ __device__ inline SmemPlan smem_plan(int kc, int nsplit, bool fp8, int dv) {
  SmemPlan s;
  const size_t eb = fp8 ? 1 : 2;
  s.q = 0;
  s.k = eb * static_cast<size_t>(kTile);
  s.vt = s.k + static_cast<size_t>(kc) * 128 * eb;
  s.pm = s.vt + static_cast<size_t>(kblocks(kc, fp8)) * dv * 128;
  // the chunk's value rows are staged after V^T before their transpose (the wide slice
  // gathers them from global memory instead: no room)
  const size_t main_end = s.pm + (kc == kWideKc ? 0 : static_cast<size_t>(kblocks(kc, fp8)) * kTile);
  const int rows_per = (kRows + nsplit - 1) / nsplit;
  const size_t recv_bytes = static_cast<size_t>(nsplit) * rows_per * dv * 4;
  const size_t stage_bytes = static_cast<size_t>(kRows) * dv * 4;
  size_t end = main_end;
  // this CTA's O share is staged in V^T and P (dead once P V completed) when they are
  // large enough; the O receive buffer reuses Q and K (dead once every CTA passed the
  // statistics exchange) when they are large enough; else each follows the tiles
  if (main_end - s.vt >= stage_bytes) {
    s.stage = s.vt;
  } else {
    s.stage = (end + 1023) / 1024 * 1024;
    end = s.stage + stage_bytes;
  }
  if (recv_bytes <= s.vt) {
    s.recv = 0;
  } else {
    s.recv = (end + 1023) / 1024 * 1024;
    end = s.recv + recv_bytes;
  }
  s.stats = (end + 15) / 16 * 16;                            // [kMaxSplit][128] float2
  s.part = s.stats + static_cast<size_t>(kMaxSplit) * kRows * 8;   // [parts][128] float2
  s.bar = s.part + static_cast<size_t>(attn_threads(kc) / 128) * kRows * 8;
  s.total = s.bar + 64;
  return s;
}

// kDv: head dims of O per CTA (the P V contraction's N): kDh, or kDh / 2 when the two
// halves run as two CTAs that repeat S and the softmax (small grids, where the O
// exchange through distributed shared memory dominates)
template <int KC, bool kF8, int kDv>
__global__ void __launch_bounds__(attn_threads(KC)) attn_kernel(const KParams p) {
  constexpr int kThreads = attn_threads(KC);
  constexpr int kParts = kThreads / 128;        // warps (key parts) per TMEM lane quarter
  constexpr bool kStageV = KC != kWideKc;       // chunk values staged in shared memory (else gathered)
  static_assert(KC != kWideKc || (!kF8 && kDv == kDh), "the wide slice: bf16, all head dims");
  constexpr int kTileV = kDv * 128;   // bytes of one [kDv rows][128 B] block of V^T
  constexpr int kDsplit = kDh / kDv;
  constexpr int kPart = KC / kParts;            // keys of the slice handled by one thread of a row
  constexpr int kBlk = kF8 ? (KC + 127) / 128 : KC / 64;   // key blocks of the P V contraction
  constexpr int kKcp = kF8 ? kBlk * 128 : KC;   // keys of the P V contraction (E4M3: zero padded)
  constexpr int kRowChunks = kF8 ? 8 : 16;      // 16-byte chunks of one Dh-wide row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemPlan sp = smem_plan(KC, p.nsplit, kF8, kDv);
  // S done, O done, every slice's statistics received, this CTA's O band received
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + sp.bar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 4);
  float2* sStats = reinterpret_cast<float2*>(smem + sp.stats);  // [rank][row] (slice max, slice sum)
  float2* sPart = reinterpret_cast<float2*>(smem + sp.part);    // [part][row]
  float* recv = reinterpret_cast<float*>(smem + sp.recv);       // [rank][local row][128]
  __shared__ int s_abort;

  const int split = blockIdx.x;
  const int qt = blockIdx.y;
  const int g = blockIdx.z / kDsplit;              // KV head
  const int d0 = (blockIdx.z % kDsplit) * kDv;     // this CTA's head dims of O: [d0, d0 + kDv)
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, part = warp >> 2;
  const bool tl_on = p.tl != nullptr && tid == 0;
  __shared__ uint64_t tt[kTlStamps];   // timeline stamps (thread 0)
  if (tl_on)
    for (int i = 0; i < kTlStamps; ++i) tt[i] = 0;
  if (tl_on) tt[0] = global_ns();
  const int nkeys = p.P + p.M;
  const int t0 = split * KC;
  const int nvalid = min(KC, nkeys - t0);
  // TMEM columns: S = Q K^T [0, KC), O [KC, KC + kDv), P from kPcol0 (the A operand of
  // P V: two bf16 or four E4M3 probabilities of a row per 32-bit column)
  constexpr int kPcol0 = KC + kDv;
  constexpr int kPcols = kF8 ? kKcp / 4 : KC / 2;
  static_assert(kPcol0 + kPcols <= 512, "S, O and P must fit in tensor memory");
  constexpr uint32_t ncols = (kPcol0 + kPcols) <= 256 ? 256u : 512u;
  const int rows_per = (kRows + p.nsplit - 1) / p.nsplit;
  const int tile_rows = min(kRows, p.G * p.M - qt * kRows);   // real (head, row) rows of the tile
  // rows [lo, hi) of the band finalised by cluster rank o (empty past the real rows)
  auto band = [&](int o, int& lo, int& hi) {
    lo = o * rows_per;
    hi = min(min(kRows, lo + rows_per), tile_rows);
    if (hi < lo) hi = lo;
  };
  // static scales (set through the host API, never by a kernel of the decision):
  // fetched at the start, off the critical path
  // log2(e) / sqrt(Dh), times the E4M3 codes' dequantisation fp32(s_q * s_k)
  const float kscale = 1.4426950408889634f * rsqrtf(static_cast<float>(kDh)) *
                       (kF8 ? __fmul_rn(p.s_qkv[0], p.s_qkv[1]) : 1.0f);
  // E4M3 output: the reciprocal of its static scale; four-bit output: the tensor scale
  const float rs = p.out_fp8 ? (p.out_fp8 == kQNvfp4AsF16 ? *p.s_out : 1.0f / *p.s_out) : 1.0f;
  const float dv = kF8 ? __fdiv_rn(p.s_qkv[2], 448.0f) : 1.0f;   // E4M3 P and V: fp32(s_v / 448)

  if (tid == 0) {
    s_abort = 0;
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_init(&bar[2], 1);
    mbar_init(&bar[3], 1);
    fence_mbar_init();
    // every slice pushes (max, sum) of all 128 rows; this CTA's band of O arrives from
    // every slice by bulk copies
    mbar_arrive_expect_tx(&bar[2], static_cast<uint32_t>(p.nsplit * kRows * 8));
    int lo, hi;
    band(static_cast<int>(cluster_rank()), lo, hi);
    mbar_arrive_expect_tx(&bar[3], static_cast<uint32_t>(p.nsplit * (hi - lo) * kDv * 4));
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
  pdl_trigger();   // after TMEM is held: a later GEMM waiting on this grid cannot starve it

  const uint32_t base = smem_u32(smem);
  const uint32_t sQa = base + sp.q, sKa = base + sp.k, sVta = base + sp.vt, sPa = base + sp.pm;

  // ---- prefix keys and transposed values of this slice (written before this graph ran)
  for (int idx = tid; idx < KC * kRowChunks; idx += kThreads) {
    const int i = idx / kRowChunks, c16 = idx % kRowChunks;   // key row, 16-byte chunk of it
    const int t = t0 + i;
    const uint32_t dst = sKa + (c16 >> 3) * (KC * 128) + swz(i, c16 & 7);
    if (t < p.P) {
      if constexpr (kF8)
        cp_async16(dst, p.kpre8 + (static_cast<size_t>(t) * p.Hkv + g) * kDh + c16 * 16);
      else
        cp_async16(dst, p.kpre + (static_cast<size_t>(t) * p.Hkv + g) * kDh + c16 * 8);
    } else if (t >= nkeys) {
      st_shared_v4(dst, make_uint4(0, 0, 0, 0));
    }
  }
  // V^T rows of this CTA's head dims: eight threads per row copy 16 bytes at a time. The
  // cache row is padded with zeros from P to P_pad, so a group straddling the end of
  // the prefix is copied whole; its keys >= P are overwritten with the chunk's values.
  if constexpr (kF8) {   // E4M3: 16 keys per 16-byte group; the padding keys [KC, kKcp) are zero
    const int d = tid & (kDv - 1);
    const uint8_t* vrow = p.vtpre8 + (static_cast<size_t>(g) * kDh + d0 + d) * p.p16;
    for (int grp = tid / kDv; grp < kKcp / 16; grp += kThreads / kDv) {
      const int t = t0 + grp * 16;
      const uint32_t dst = sVta + (grp >> 3) * kTileV + swz(d, grp & 7);
      if (grp * 16 < KC && t < p.P)
        cp_async16(dst, vrow + t);
      else
        st_shared_v4(dst, make_uint4(0, 0, 0, 0));
    }
  } else {
    const int d = tid & (kDv - 1);
    const __nv_bfloat16* vrow = p.vtpre + (static_cast<size_t>(g) * kDh + d0 + d) * p.p_pad;
    for (int grp = tid / kDv; grp < KC / 8; grp += kThreads / kDv) {
      const int t = t0 + grp * 8;
      const uint32_t dst = sVta + (grp >> 3) * kTileV + swz(d, grp & 7);
      if (t < p.P)
        cp_async16(dst, vrow + t);
      else
        st_shared_v4(dst, make_uint4(0, 0, 0, 0));
    }
  }
  cp_async_commit();
  pdl_wait();   // Q, K, V of the chunk are written by the QKV GEMM
  if (tl_on) tt[1] = global_ns();

  // ---- stacked query rows and the chunk's own keys (rows P..P+M-1 of the key axis)
  for (int idx = tid; idx < kRows * kRowChunks; idx += kThreads) {
    const int r = idx / kRowChunks, c16 = idx % kRowChunks;
    const int R = qt * kRows + r;
    const uint32_t dst = sQa + (c16 >> 3) * kTile + swz(r, c16 & 7);
    if (R < p.G * p.M) {
      const int hl = R / p.M, m = R % p.M;
      if constexpr (kF8)
        cp_async16(dst, p.qkv8 + static_cast<size_t>(m) * p.ldq + (g * p.G + hl) * kDh + c16 * 16);
      else
        cp_async16(dst, p.qkv + static_cast<size_t>(m) * p.ldq + (g * p.G + hl) * kDh + c16 * 8);
    } else {
      st_shared_v4(dst, make_uint4(0, 0, 0, 0));
    }
  }
  const int c_lo = max(t0, p.P), c_hi = min(t0 + KC, nkeys);
  const int nchunk = c_hi > c_lo ? c_hi - c_lo : 0;   // <= KC
  for (int idx = tid; idx < nchunk * kRowChunks; idx += kThreads) {
    const int t = c_lo + idx / kRowChunks, c16 = idx % kRowChunks;
    // the chunk's values are staged row-major in the P tiles, transposed below
    if constexpr (kF8) {
      const uint8_t* row = p.qkv8 + static_cast<size_t>(t - p.P) * p.ldq;
      cp_async16(sKa + swz(t - t0, c16), row + (p.H + g) * kDh + c16 * 16);
      cp_async16(sPa + static_cast<uint32_t>((t - c_lo) * kDh + c16 * 16), row + (p.H + p.Hkv + g) * kDh + c16 * 16);
    } else {
      const __nv_bfloat16* row = p.qkv + static_cast<size_t>(t - p.P) * p.ldq;
      cp_async16(sKa + (c16 >> 3) * (KC * 128) + swz(t - t0, c16 & 7), row + (p.H + g) * kDh + c16 * 8);
      if constexpr (kStageV)
        cp_async16(sPa + static_cast<uint32_t>(((t - c_lo) * kDh + c16 * 8) * 2),
                   row + (p.H + p.Hkv + g) * kDh + c16 * 8);
    }
  }
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();   // V^T groups and the staged chunk values are in place
  if (tl_on) tt[2] = global_ns();
  if (nchunk > 0) {
    // shared -> shared transpose of the chunk's values into V^T (keys along K), this
    // CTA's dims: one thread per (16-byte V^T group holding chunk keys, head dim), the
    // group's current bytes (prefix keys, zeros) merged with the chunk keys it holds,
    // gathered from the row-major staging (consecutive threads take consecutive dims),
    // and written back by one 16-byte store
    constexpr int kPer = kF8 ? 16 : 8;   // keys per 16-byte group
    const int g_lo = (c_lo - t0) / kPer, g_hi = (c_hi - 1 - t0) / kPer;
    if constexpr (!kStageV) {
      if (p.vtc) {
        // wide slice with the chunk's values already transposed: whole aligned groups of
        // 8 keys by 16-byte asynchronous copies, a straddling group merged key by key;
        // consecutive threads take consecutive groups of one dim (contiguous sources)
        const int ngrp = g_hi - g_lo + 1;
        for (int idx = tid; idx < ngrp * kDv; idx += kThreads) {
          const int d = idx / ngrp, G = g_lo + idx % ngrp;
          const int t = t0 + G * 8;
          const __nv_bfloat16* vrow = p.vtc + static_cast<size_t>(g * kDh + d0 + d) * p.m_pad;
          const size_t off = static_cast<size_t>(sp.vt) + (G >> 3) * kTileV + swz(d, G & 7);
          if (t >= c_lo && t + 8 <= c_hi && (t - p.P) % 8 == 0) {
            cp_async16(base + static_cast<uint32_t>(off), vrow + (t - p.P));
          } else {
            uint4* grp = reinterpret_cast<uint4*>(smem + off);
            uint4 u = *grp;
            uint16_t* e16 = reinterpret_cast<uint16_t*>(&u);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (t + e >= c_lo && t + e < c_hi)
                e16[e] = reinterpret_cast<const uint16_t*>(vrow)[t + e - p.P];
            *grp = u;
          }
        }
        cp_async_commit();
        cp_async_wait_all();
      }
    }
    if constexpr (!kStageV) if (!p.vtc) {
      // wide slice: every (group, dim) task of this thread loads its keys' values from
      // the QKV output first (all loads in flight together, two values per register),
      // then merges them into the groups
      constexpr int kTasks = (KC / 8) * kDv / kThreads;
      const int ntask = (g_hi - g_lo + 1) * kDv;
      const uint16_t* vbase = reinterpret_cast<const uint16_t*>(p.qkv) + (p.H + p.Hkv + g) * kDh + d0;
      uint32_t w[kTasks][4];
#pragma unroll
      for (int i = 0; i < kTasks; ++i) {
        const int idx = tid + i * kThreads;
        const int d = idx % kDv, G = g_lo + idx / kDv;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const int t = t0 + G * 8 + e;
          const uint32_t lo = idx < ntask && t >= c_lo && t < c_hi ? vbase[static_cast<size_t>(t - p.P) * p.ldq + d] : 0u;
          const uint32_t hi =
              idx < ntask && t + 1 >= c_lo && t + 1 < c_hi ? vbase[static_cast<size_t>(t + 1 - p.P) * p.ldq + d] : 0u;
          w[i][e / 2] = lo | (hi << 16);
        }
      }
#pragma unroll
      for (int i = 0; i < kTasks; ++i) {
        const int idx = tid + i * kThreads;
        if (idx >= ntask) break;
        const int d = idx % kDv, G = g_lo + idx / kDv;
        uint4* grp = reinterpret_cast<uint4*>(smem + sp.vt + (G >> 3) * kTileV + swz(d, G & 7));
        uint4 u = *grp;
        uint16_t* e16 = reinterpret_cast<uint16_t*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int t = t0 + G * 8 + e;
          if (t >= c_lo && t < c_hi) e16[e] = static_cast<uint16_t>(w[i][e / 2] >> (16 * (e & 1)));
        }
        *grp = u;
      }
    }
    for (int idx = tid; kStageV && idx < (g_hi - g_lo + 1) * kDv; idx += kThreads) {
      const int d = idx % kDv, G = g_lo + idx / kDv;
      uint4* grp = reinterpret_cast<uint4*>(smem + sp.vt + (G >> 3) * kTileV + swz(d, G & 7));
      uint4 u = *grp;
      if constexpr (kF8) {
        uint8_t* e8 = reinterpret_cast<uint8_t*>(&u);
        const uint8_t* vstage = smem + sp.pm;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int t = t0 + G * 16 + e;
          if (t >= c_lo && t < c_hi) e8[e] = vstage[(t - c_lo) * kDh + d0 + d];
        }
      } else {
        uint16_t* e16 = reinterpret_cast<uint16_t*>(&u);
        const uint16_t* vstage = reinterpret_cast<const uint16_t*>(smem + sp.pm);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int t = t0 + G * 8 + e;
          if (t >= c_lo && t < c_hi) e16[e] = vstage[(t - c_lo) * kDh + d0 + d];
        }
      }
      *grp = u;
    }
  }
  fence_async_smem();   // generic-proxy shared-memory writes -> tensor-core reads
  __syncthreads();
  if (tl_on) tt[3] = global_ns();

  // ---- S = Q K^T into TMEM columns [0, KC)
  if (tid == 0) {
    tc_fence_after();
    const uint32_t idesc = make_idesc(kF8, kRows, static_cast<uint32_t>(KC));
#pragma unroll
    for (int b = 0; b < (kF8 ? 1 : 2); ++b) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc_mma<kF8>(tmem, sw128_kmajor_desc(sQa + b * kTile + k * 32),
                    sw128_kmajor_desc(sKa + b * (KC * 128) + k * 32), idesc, (b | k) ? 1u : 0u);
    }
    tc_commit(&bar[0]);
  }
  if (!mbar_wait(&bar[0], 0)) {
    atomicOr(p.err, kErrPipelineTimeout);
    s_abort = 1;
  }
  if (tl_on) tt[4] = global_ns();
  tc_fence_after();
  __syncwarp();

  const int r = quarter * 32 + lane;   // this thread's row == its TMEM lane
  const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  const int c0 = part * kPart;         // this thread's keys: [c0, c0 + kPart) of the slice

  // ---- pass 1: this row part's scores (kept in registers), max and sum of exp
  float sv[kPart];
#pragma unroll
  for (int c = 0; c + 32 <= kPart; c += 32) {   // 32 columns per TMEM load
    float v[32];
    tmem_ld32(t_row + static_cast<uint32_t>(c0 + c), v);
#pragma unroll
    for (int e = 0; e < 32; ++e) sv[c + e] = c0 + c + e < nvalid ? v[e] * kscale : -INFINITY;
  }
  if constexpr (kPart % 32 != 0) {
    constexpr int c = kPart - 16;
    float v[16];
    tmem_ld16(t_row + static_cast<uint32_t>(c0 + c), v);
#pragma unroll
    for (int e = 0; e < 16; ++e) sv[c + e] = c0 + c + e < nvalid ? v[e] * kscale : -INFINITY;
  }
  float mh = -INFINITY;
#pragma unroll
  for (int e = 0; e < kPart; ++e) mh = fmaxf(mh, sv[e]);
  // sv <- exp(s - m_part): the only exponentials of the row; pass 2 rescales them
  float lh = 0.f;
#pragma unroll
  for (int e = 0; e < kPart; ++e) {
    sv[e] = mh > -INFINITY ? ex2_approx(sv[e] - mh) : 0.f;
    lh += sv[e];
  }
  sPart[part * kRows + r] = make_float2(mh, lh);
  if (tl_on) tt[5] = global_ns();
  __syncthreads();
  // the slice statistics of row r, pushed to every CTA of the cluster (slot = own rank)
  cluster_wait();   // every peer has started: its shared memory exists
  if (tl_on) tt[6] = global_ns();
  if (part == 0) {
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < kParts; ++q) m = fmaxf(m, sPart[q * kRows + r].x);
    float l = 0.f;
#pragma unroll
    for (int q = 0; q < kParts; ++q) {
      const float2 st = sPart[q * kRows + r];
      l += st.y > 0.f ? st.y * ex2_approx(st.x - m) : 0.f;
    }
    const uint32_t rank = cluster_rank();
    const uint32_t off = smem_u32(sStats + rank * kRows + r);
    const uint32_t mb = smem_u32(&bar[2]);
    for (int q = 0; q < p.nsplit; ++q)
      st_async_v2(map_dsmem(off, static_cast<uint32_t>(q)), m, l, map_dsmem(mb, static_cast<uint32_t>(q)));
    if (tl_on) tt[7] = global_ns();
  }
  // Every slice's statistics have landed. Each peer sent them after its S = Q K^T
  // completed, so from here on its Q and K tiles are dead and may receive O shares.
  if (!mbar_wait(&bar[2], 0)) {
    atomicOr(p.err, kErrPipelineTimeout);
    s_abort = 1;
  }
  if (tl_on) tt[8] = global_ns();
  // the row's global max and 1 / sum in slice order, by every thread of the row (the
  // same operations in the same order in each, so no hand-off through shared memory);
  // its rescaling exponentials, like pass 1's, by the approximate 2^x: they only feed
  // probabilities rounded to bf16 or E4M3 (the accurate exp2f kept this phase 0.2 us
  // longer per layer-step)
  float gmax, ginv;
  {
    float2 st[kMaxSplit];
#pragma unroll
    for (int q = 0; q < kMaxSplit; ++q) st[q] = q < p.nsplit ? sStats[q * kRows + r] : make_float2(-INFINITY, 0.f);
    float gm = -INFINITY;
#pragma unroll
    for (int q = 0; q < kMaxSplit; ++q) gm = fmaxf(gm, st[q].x);
    float gs = 0.f;
#pragma unroll
    for (int q = 0; q < kMaxSplit; ++q)
      if (q < p.nsplit) gs += st[q].y * ex2_approx(st[q].x - gm);
    gmax = gm;
    ginv = 1.0f / gs;
  }

  // ---- pass 2: P = bf16(exp(s - m_part) * exp(m_part - M) / L) into tensor memory,
  // each thread its row's keys [c0, c0 + kPart): the A operand of P V
  const float fscale = mh > -INFINITY ? ex2_approx(mh - gmax) * ginv : 0.f;
  {
    constexpr int kPc = kF8 ? kPart / 4 : kPart / 2;   // this thread's P columns
    uint32_t pw[kPc];
    if constexpr (kF8) {
      // E4M3 probabilities with static scale 1/448: code = E4M3(P * 448), four keys per column
#pragma unroll
      for (int c = 0; c < kPc; ++c) {
        uint32_t packed = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kk = 4 * c + e;
          const float pv = c0 + kk < nvalid ? sv[kk] * fscale : 0.f;
          packed |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(pv * 448.0f, __NV_SATFINITE, __NV_E4M3)) << (8 * e);
        }
        pw[c] = packed;
      }
    } else {
#pragma unroll
      for (int c = 0; c < kPc; ++c) {
        const int kk = 2 * c;
        pw[c] = pack_bf16(c0 + kk < nvalid ? sv[kk] * fscale : 0.f, c0 + kk + 1 < nvalid ? sv[kk + 1] * fscale : 0.f);
      }
    }
    tmem_st_cols<kPc>(t_row + static_cast<uint32_t>(kPcol0 + c0 / (kF8 ? 4 : 2)), pw);
    if constexpr (kF8) {   // the zero-padded keys [KC, kKcp): four columns per 16 keys
      const uint32_t zero[4] = {0u, 0u, 0u, 0u};
      for (int j = part; j < (kKcp - KC) / 16; j += kParts)
        tmem_st4(t_row + static_cast<uint32_t>(kPcol0 + (KC + j * 16) / 4), zero);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  if (tl_on) tt[9] = global_ns();

  // ---- O = P V into TMEM columns [KC, KC + kDv): this CTA's head dims
  if (tid == 0) {
    tc_fence_after();
    const uint32_t idesc = make_idesc(kF8, kRows, kDv);
#pragma unroll
    for (int b = 0; b < kBlk; ++b) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc_mma_ts<kF8>(tmem + static_cast<uint32_t>(KC), tmem + static_cast<uint32_t>(kPcol0 + b * 32 + k * 8),
                       sw128_kmajor_desc(sVta + b * kTileV + k * 32), idesc, (b | k) ? 1u : 0u);
    }
    tc_commit(&bar[1]);
  }
  if (!mbar_wait(&bar[1], 0)) {
    atomicOr(p.err, kErrPipelineTimeout);
    s_abort = 1;
  }
  if (tl_on) tt[10] = global_ns();
  tc_fence_after();
  __syncwarp();

  // ---- this slice's share of O (already normalised by the global sum) goes band by
  // band to the CTA that finalises it (rows are split into bands of rows_per). TMEM
  // gives each thread one row, so the share is first staged row-major in shared
  // memory (16-byte chunks swizzled by row: conflict-free); then one bulk copy per
  // band moves the band's rows into the owner's receive slot for this rank, counted
  // on the owner's mbarrier (one lane per band issues its copy: a single thread
  // issuing them in turn took twice as long).
  {
    constexpr int kCols = kDv / kParts;   // O columns read by one thread
    constexpr int kRowBytes = kDv * 4;    // one staged row of this CTA's O share
    const uint32_t stage = base + static_cast<uint32_t>(sp.stage);
#pragma unroll
    for (int c = 0; c < kCols; c += 16) {
      float v[16];
      tmem_ld16(t_row + static_cast<uint32_t>(KC + part * kCols + c), v);
#pragma unroll
      for (int e = 0; e < 16; e += 4) {
        const int chunk = (part * kCols + c + e) >> 2;   // 16-byte chunk (0..kDv/4-1) of the row
        st_shared_v4(stage + r * kRowBytes + ((chunk ^ (r & 7)) << 4),
                     make_uint4(__float_as_uint(v[e]), __float_as_uint(v[e + 1]), __float_as_uint(v[e + 2]),
                                __float_as_uint(v[e + 3])));
      }
    }
    fence_async_smem();   // the staged rows -> the bulk copies' reads
    __syncthreads();
    static_assert(kThreads / 32 >= kMaxSplit, "a warp for every band");
    if (lane == 0 && warp < p.nsplit) {   // band o's copy issued by warp o (in parallel)
      const int o = warp;
      const uint32_t slot = smem_u32(recv + static_cast<size_t>(cluster_rank()) * rows_per * kDv);
      int lo, hi;
      band(o, lo, hi);
      if (hi > lo)
        bulk_copy_to_peer(map_dsmem(slot, static_cast<uint32_t>(o)), stage + static_cast<uint32_t>(lo * kRowBytes),
                          static_cast<uint32_t>((hi - lo) * kRowBytes),
                          map_dsmem(smem_u32(&bar[3]), static_cast<uint32_t>(o)));
    }
    if (tl_on) tt[11] = global_ns();
  }
  if (!mbar_wait(&bar[3], 0)) {   // every slice's share of this CTA's band has landed
    atomicOr(p.err, kErrPipelineTimeout);
    s_abort = 1;
  }
  if (tl_on) tt[12] = global_ns();
  // Once every owner has its band, no bulk copy still reads this CTA's stage: each
  // CTA arrives here and waits before exit (lifetime only; the data is ordered by
  // the mbarriers).
  cluster_arrive_relaxed();

  // ---- sum the slices' shares in fixed slice order, quantise, store
  if (s_abort == 0) {
    const int rank = static_cast<int>(cluster_rank());
    // kDv / 4 lanes per row, 4 head dims each
    constexpr int kLanesRow = kDv / 4;
    constexpr int kRowsWarp = 32 / kLanesRow;
    const int l16 = lane % kLanesRow;
    const int e4 = l16 * 4;
    for (int lr = warp * kRowsWarp + lane / kLanesRow; lr < rows_per; lr += (kThreads / 32) * kRowsWarp) {
      const int rr = rank * rows_per + lr;
      const int R = qt * kRows + rr;
      if (rr >= kRows || R >= p.G * p.M) break;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      const int sw = (l16 ^ (rr & 7)) << 2;   // the staged row's swizzled chunk
      // slots in groups of four whose loads are issued together, summed in slot order
      for (int q0 = 0; q0 < p.nsplit; q0 += 4) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int q = q0 + j < p.nsplit ? q0 + j : q0;
          v[j] = *reinterpret_cast<const float4*>(recv + (q * rows_per + lr) * kDv + sw);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (q0 + j < p.nsplit) {
            acc.x += v[j].x;
            acc.y += v[j].y;
            acc.z += v[j].z;
            acc.w += v[j].w;
          }
        }
      }
      if constexpr (kF8) {
        acc.x *= dv;
        acc.y *= dv;
        acc.z *= dv;
        acc.w *= dv;
      }
      const int hl = R / p.M, m = R % p.M;
      const size_t oidx = static_cast<size_t>(m) * (p.H * kDh) + (g * p.G + hl) * kDh + d0 + e4;
      if (p.out_fp8 == kQNvfp4AsF16) {
        // four-bit output: a 16-dim block is four consecutive lanes of this row (the row's
        // lanes run the loop together: mask them)
        const unsigned rmask = kLanesRow == 32 ? 0xffffffffu : (0xffffu << (lane & 16));
        float a = fmaxf(fmaxf(fabsf(acc.x), fabsf(acc.y)), fmaxf(fabsf(acc.z), fabsf(acc.w)));
        a = fmaxf(a, __shfl_xor_sync(rmask, a, 1));
        a = fmaxf(a, __shfl_xor_sync(rmask, a, 2));
        float den;
        const float bs = nvfp4_block(a, rs, &den);
        const __half2 lo = nvfp4_pair(acc.x, acc.y, bs, den), hi = nvfp4_pair(acc.z, acc.w, bs, den);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&lo);
        u.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(static_cast<__half*>(p.out) + oidx) = u;
      } else if (p.out_fp8) {
        uchar4 cc;
        cc.x = static_cast<uint8_t>(__nv_cvt_float_to_fp8(acc.x * rs, __NV_SATFINITE, __NV_E4M3));
        cc.y = static_cast<uint8_t>(__nv_cvt_float_to_fp8(acc.y * rs, __NV_SATFINITE, __NV_E4M3));
        cc.z = static_cast<uint8_t>(__nv_cvt_float_to_fp8(acc.z * rs, __NV_SATFINITE, __NV_E4M3));
        cc.w = static_cast<uint8_t>(__nv_cvt_float_to_fp8(acc.w * rs, __NV_SATFINITE, __NV_E4M3));
        if (p.out_fp8 == kQFp8AsF16) {   // the codes' f16 values (exact)
          const uint8_t b[4] = {cc.x, cc.y, cc.z, cc.w};
          uint32_t h[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            h[i] = __half_as_ushort(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b[i]), __NV_E4M3)));
          *reinterpret_cast<uint2*>(static_cast<__half*>(p.out) + oidx) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
        } else {
          *reinterpret_cast<uchar4*>(static_cast<uint8_t*>(p.out) + oidx) = cc;
        }
      } else {
        uint2 u;
        u.x = pack_bf16(acc.x, acc.y);
        u.y = pack_bf16(acc.z, acc.w);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + oidx) = u;
      }
    }
  }
  if (tl_on) tt[13] = global_ns();
  cluster_wait();   // every owner has its band: no copy still reads this CTA
  tc_fence_before();
  __syncthreads();
  if (tl_on) {
    tt[14] = global_ns();
    tl_record(p.tl, kTlAttn, gridDim.y * gridDim.z, blockIdx.y * gridDim.z + blockIdx.z, tt);
  }
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

size_t attn_smem_bytes(int kc, int nsplit, int fp8, int dv) {
  return 1024 + smem_plan(kc, nsplit, fp8 != 0, dv).total;
}

namespace {

const void* attn_kernel_for(int kc, bool fp8, int dv) {
  const bool half = dv == kDh / 2;
  switch ((kc * 2 + (fp8 ? 1 : 0)) * 2 + (half ? 1 : 0)) {
    case 256: return reinterpret_cast<const void*>(attn_kernel<64, false, kDh>);
    case 512: return reinterpret_cast<const void*>(attn_kernel<128, false, kDh>);
    case 768: return reinterpret_cast<const void*>(attn_kernel<192, false, kDh>);
    case 1024: return reinterpret_cast<const void*>(attn_kernel<kWideKc, false, kDh>);
    case 258: return reinterpret_cast<const void*>(attn_kernel<64, true, kDh>);
    case 514: return reinterpret_cast<const void*>(attn_kernel<128, true, kDh>);
    case 770: return reinterpret_cast<const void*>(attn_kernel<192, true, kDh>);
    case 257: return reinterpret_cast<const void*>(attn_kernel<64, false, kDh / 2>);
    case 513: return reinterpret_cast<const void*>(attn_kernel<128, false, kDh / 2>);
    case 769: return reinterpret_cast<const void*>(attn_kernel<192, false, kDh / 2>);
    case 259: return reinterpret_cast<const void*>(attn_kernel<64, true, kDh / 2>);
    case 515: return reinterpret_cast<const void*>(attn_kernel<128, true, kDh / 2>);
    case 771: return reinterpret_cast<const void*>(attn_kernel<192, true, kDh / 2>);
    default: return nullptr;
  }
}

}  // namespace

int attn_clusters_per_wave(int kc, int nsplit, int fp8, int dv) {
  const void* k = attn_kernel_for(kc, fp8 != 0, dv);
  if (!k || nsplit < 1 || nsplit > kMaxSplit || attn_configure() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nsplit), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(attn_threads(kc)), 1, 1);
  cfg.dynamicSmemBytes = attn_smem_bytes(kc, nsplit, fp8, dv);
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeClusterDimension;
  at.val.clusterDim.x = static_cast<unsigned>(nsplit);
  at.val.clusterDim.y = 1;
  at.val.clusterDim.z = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
    cudaGetLastError();   // a failed query is not an error of the caller's next call
    return 0;
  }
  return n;
}

int attn_plan_launch(int M, int P, int G, int Hkv, int fp8, int sms, int* kc, int* nsplit) {
  const int st = attn_plan(M, P, kc, nsplit);
  if (st != FM_OK || fp8) return st;
  const int tiles = (G * M + kRows - 1) / kRows;
  if (4 * *nsplit * tiles * Hkv <= sms) return FM_OK;   // the small grids (head dims split in two)
  const int keys = P + M;
  const int ns_w = (keys + kWideKc - 1) / kWideKc;
  if (ns_w > kMaxSplit) return FM_OK;
  // the wide slice when its clusters (fewer CTAs each) need fewer waves of the GPU
  const int per0 = attn_clusters_per_wave(*kc, *nsplit, 0, kDh), per1 = attn_clusters_per_wave(kWideKc, ns_w, 0, kDh);
  if (per0 <= 0 || per1 <= 0) return FM_OK;
  const int clusters = tiles * Hkv;
  if ((clusters + per1 - 1) / per1 < (clusters + per0 - 1) / per0) {
    *kc = kWideKc;
    *nsplit = ns_w;
  }
  return FM_OK;
}

namespace {

cudaError_t attn_configure_impl() {
  const void* ks[13] = {reinterpret_cast<const void*>(attn_kernel<kWideKc, false, kDh>),
                        reinterpret_cast<const void*>(attn_kernel<64, false, kDh>),
                        reinterpret_cast<const void*>(attn_kernel<128, false, kDh>),
                        reinterpret_cast<const void*>(attn_kernel<192, false, kDh>),
                        reinterpret_cast<const void*>(attn_kernel<64, true, kDh>),
                        reinterpret_cast<const void*>(attn_kernel<128, true, kDh>),
                        reinterpret_cast<const void*>(attn_kernel<192, true, kDh>),
                        reinterpret_cast<const void*>(attn_kernel<64, false, kDh / 2>),
                        reinterpret_cast<const void*>(attn_kernel<128, false, kDh / 2>),
                        reinterpret_cast<const void*>(attn_kernel<192, false, kDh / 2>),
                        reinterpret_cast<const void*>(attn_kernel<64, true, kDh / 2>),
                        reinterpret_cast<const void*>(attn_kernel<128, true, kDh / 2>),
                        reinterpret_cast<const void*>(attn_kernel<192, true, kDh / 2>)};
  for (const void* k : ks) {
    const cudaError_t e = allow_max_dynamic_smem(k);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t attn_configure() { return configure_once(2, attn_configure_impl); }

cudaError_t attn_launch(const AttnArgs& a, const LaunchOpts& o) {
  KParams p;
  p.qkv = a.qkv;
  p.qkv8 = reinterpret_cast<const uint8_t*>(a.qkv);
  p.kpre8 = a.kpre8;
  p.vtpre8 = a.vtpre8;
  p.p16 = a.p16;
  p.s_qkv = a.s_qkv;
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
  p.vtc = a.vtc;
  p.m_pad = a.m_pad;
  if (a.vtc && (a.m_pad < a.M || a.m_pad % 8)) return cudaErrorInvalidValue;
  p.err = a.err;
  p.tl = o.tl;
  if (a.fp8 && (!a.kpre8 || !a.vtpre8 || !a.s_qkv || a.p16 % 16)) return cudaErrorInvalidValue;
  const int rows = p.G * p.M;
  const int tiles = (rows + kRows - 1) / kRows;
  // The two halves of O's head dims become two CTAs (repeating S and the softmax) while
  // the doubled grid still fits in one wave on half the SMs; larger grids keep one CTA.
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
      sms = 148;
  }
  const bool dsplit = a.kc != kWideKc && 4 * a.nsplit * tiles * a.Hkv <= sms;
  // z: KV head x (with the split) the two halves of the head dims of O
  const dim3 grid(static_cast<unsigned>(a.nsplit), static_cast<unsigned>(tiles),
                  static_cast<unsigned>(a.Hkv * (dsplit ? 2 : 1)));
  LaunchOpts lo = o;
  lo.cluster = dim3(static_cast<unsigned>(a.nsplit), 1, 1);
  const size_t smem = attn_smem_bytes(a.kc, a.nsplit, a.fp8, dsplit ? kDh / 2 : kDh);
  const dim3 blk(static_cast<unsigned>(attn_threads(a.kc)));
  switch ((a.kc * 2 + (a.fp8 ? 1 : 0)) * 2 + (dsplit ? 1 : 0)) {
    case 256: return launch(attn_kernel<64, false, kDh>, grid, blk, smem, lo, p);
    case 512: return launch(attn_kernel<128, false, kDh>, grid, blk, smem, lo, p);
    case 768: return launch(attn_kernel<192, false, kDh>, grid, blk, smem, lo, p);
    case 1024: return launch(attn_kernel<kWideKc, false, kDh>, grid, blk, smem, lo, p);
    case 258: return launch(attn_kernel<64, true, kDh>, grid, blk, smem, lo, p);
    case 514: return launch(attn_kernel<128, true, kDh>, grid, blk, smem, lo, p);
    case 770: return launch(attn_kernel<192, true, kDh>, grid, blk, smem, lo, p);
    case 257: return launch(attn_kernel<64, false, kDh / 2>, grid, blk, smem, lo, p);
    case 513: return launch(attn_kernel<128, false, kDh / 2>, grid, blk, smem, lo, p);
    case 769: return launch(attn_kernel<192, false, kDh / 2>, grid, blk, smem, lo, p);
    case 259: return launch(attn_kernel<64, true, kDh / 2>, grid, blk, smem, lo, p);
    case 515: return launch(attn_kernel<128, true, kDh / 2>, grid, blk, smem, lo, p);
    case 771: return launch(attn_kernel<192, true, kDh / 2>, grid, blk, smem, lo, p);
    default: return cudaErrorInvalidValue;
  }
}

namespace {

__global__ void prefix_quant_kernel(const __nv_bfloat16* __restrict__ kc, const __nv_bfloat16* __restrict__ vt,
                                    uint8_t* __restrict__ k8, uint8_t* __restrict__ v8t,
                                    const float* __restrict__ ascale, int P, int Hkv, int p_pad, int p16, int b,
                                    int rows, size_t nk, size_t nv) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < nk + nv;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    if (i < nk) {   // keys: [L][rows][Hkv][Dh] of the range, stored at rows b.. of [L][P][Hkv][Dh]
      const size_t per_l = static_cast<size_t>(rows) * Hkv * kDh;
      const int l = static_cast<int>(i / per_l);
      const size_t rem = i % per_l;
      const size_t idx = (static_cast<size_t>(l) * P + b) * Hkv * kDh + rem;
      const float rs = 1.0f / ascale[l * 8 + FM_SITE_K];
      k8[idx] = static_cast<uint8_t>(
          __nv_cvt_float_to_fp8(__bfloat162float(kc[idx]) * rs, __NV_SATFINITE, __NV_E4M3));
    } else {   // values, transposed: [L][Hkv][Dh] rows, tokens b..b+rows-1 of each
      const size_t j = i - nk;
      const size_t vrow = j / rows;   // l * Hkv * Dh + g * Dh + d
      const int t = b + static_cast<int>(j % rows);
      const int l = static_cast<int>(vrow / (static_cast<size_t>(Hkv) * kDh));
      const float rs = 1.0f / ascale[l * 8 + FM_SITE_V];
      v8t[vrow * p16 + t] = static_cast<uint8_t>(
          __nv_cvt_float_to_fp8(__bfloat162float(vt[vrow * p_pad + t]) * rs, __NV_SATFINITE, __NV_E4M3));
    }
  }
}

}  // namespace

cudaError_t prefix_quant_launch(const __nv_bfloat16* kcache, const __nv_bfloat16* vtcache, uint8_t* k8, uint8_t* v8t,
                                const float* ascale, int L, int P, int Hkv, int p_pad, int p16, int b, int e,
                                cudaStream_t st) {
  if (b < 0 || e > P || b >= e) return cudaErrorInvalidValue;
  const int rows = e - b;
  const size_t nk = static_cast<size_t>(L) * rows * Hkv * kDh;
  const size_t nv = static_cast<size_t>(L) * Hkv * kDh * rows;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((nk + nv + 255) / 256, 2368));
  prefix_quant_kernel<<<blocks, 256, 0, st>>>(kcache, vtcache, k8, v8t, ascale, P, Hkv, p_pad, p16, b, rows, nk, nv);
  return cudaGetLastError();
}

cudaError_t transpose_v_launch(const __nv_bfloat16* v, __nv_bfloat16* vt, int L, int rows, int Hkv, int p_pad,
                               int tok_begin, cudaStream_t st) {
  transpose_v_kernel<<<1184, 256, 0, st>>>(v, vt, L, rows, Hkv, p_pad, tok_begin);
  return cudaGetLastError();
}

}  // namespace fm
