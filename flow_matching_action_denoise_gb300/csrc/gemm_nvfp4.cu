// GEMM with NVFP4 weights on tcgen05 tensor cores, and NVFP4 weight packing.
//
// NVFP4 (news article "FlashRT-PAI", section on 4-bit inference; the world-action
// decoder's weight format): a weight W' = W diag(gamma) is stored as E2M1
// elements e, one E4M3 block scale bs per 16 consecutive K elements and one fp32
// tensor scale ts, with W' ~= e * bs * ts. The product e * bs has at most six
// significant bits and lies in [2^-10, 2688], so it is exact in f16; the
// activations are E4M3 code values, also exact in f16. The kernel therefore
// decodes e * bs into f16 tiles in shared memory and runs kind::f16 MMAs with
// fp32 accumulation: the only rounding is the fp32 accumulation itself, and ts
// joins the activation scale in the consumer's dequantisation fp32(s_a * ts).
//
// Work split (one CTA per 128 weight rows x one K slice, 12 warps). A pipeline stage
// covers `chunk` 64-element K blocks (one transaction each way: TMA transactions
// and barrier round trips, not bytes, bound the per-SM streaming rate here):
//   thread 0    - producer: one bulk copy of the stage's packed weight blocks
//                 (4.5 KB per block: codes + block scales) into a raw ring, issued
//                 before the programmatic-dependent-launch wait, and one 3-D TMA
//                 box of the stage's f16 activation K blocks after it;
//   thread 32   - MMA issuer: 4 x (M=128, N=M_pad, K=16) per 64-element block;
//   warps 4..11 - decoders: two threads per weight row, each expanding half of the
//                 row's 64 elements of a block into the 128-byte-swizzled K-major
//                 f16 operand tile (eight warps: the expansion, not the tensor pipe,
//                 bounds these GEMMs; the code also takes four threads per row);
//   all warps   - epilogue: TMEM -> fp32 partial planes, or (single K slice,
//                 gate|up weight) GeGLU + static E4M3 (or four-bit) quantisation.

#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace fm {

namespace {

constexpr int kThreads = 384;                                 // 12 warps: roles, 8 decoders, epilogue
constexpr int kDecoders = kThreads - 128;                     // warps 4-11 expand the weight codes
constexpr int kDecoderWarps = kDecoders / 32;
constexpr int kRowParts = kDecoders / 128;                    // decoder threads per weight row
constexpr int kChunksPer = 8 / kRowParts;                     // 8-element chunks of a block row per thread
static_assert(kRowParts == 2 || kRowParts == 4, "two or four decoder threads per weight row");
constexpr int kTileN = 128;                                   // weight rows per CTA (MMA M)
constexpr int kKb = 64;                                       // K elements per pipeline block
constexpr int kCodeBytes = kTileN * kKb / 2;                  // 4096: two E2M1 codes per byte
constexpr int kRawBytes = kCodeBytes + kTileN * kKb / 16;     // + 512 block scales = 4608
constexpr int kMaxRawStages = 8;
constexpr int kMaxOpStages = 6;
constexpr int kATileBytes = kTileN * 128;                     // f16 [128][64], one swizzle row per weight row
constexpr size_t kSmemCap = 222 * 1024;
constexpr int kNumBars = 2 * kMaxRawStages + 3 * kMaxOpStages + 1;

struct NvParams {
  const uint8_t* wpk;   // packed blocks [N/128][K/64][kRawBytes]
  float* out;           // fp32 partial planes [s][M][N] (unscaled), or
  __half* out_geglu;    // (s == 1, gate|up interleaved by 16) f16 values of E4M3(gelu(g) u / s_q) [M][N/2]
  const float* sa;
  const float* sw;
  const float* sq;
  int geglu_nvfp4;      // out_geglu holds four-bit activation values e * bs (tensor scale *sq)
  int M, N;
  int nkb_total, nkb_cta;
  int n_pad, op_stages, raw_stages, chunk;
  int* err;
  // diagnostic timeline (nullptr = off): entry, after the PDL wait, MMAs complete,
  // outputs written, exit
  unsigned long long* tl;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline uint32_t pow2_at_least(uint32_t v, uint32_t lo) {
  uint32_t p = lo;
  while (p < v) p <<= 1;
  return p;
}

__device__ __forceinline__ uint32_t half2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Four E2M1 pairs (one byte each, element 2i in the low nibble) times the block
// scale: eight f16 values, exact.
__device__ __forceinline__ uint4 decode8(uint32_t codes4, __half2 bs2) {
  uint4 o;
  uint32_t* w = &o.x;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw r = __nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>((codes4 >> (8 * i)) & 0xffu),
                                                      __NV_E2M1);
    w[i] = half2_bits(__hmul2(__half2(r), bs2));
  }
  return o;
}

__device__ __forceinline__ __half e4m3_half(uint8_t code) {
  return __half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3));
}

__global__ void __launch_bounds__(kThreads) nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                                                              const NvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(smem_raw), 1024));
  __shared__ int s_abort;
  __shared__ int s_raw_issued, s_act_issued;

  const int S = p.op_stages, R = p.raw_stages, C = p.chunk;
  const uint32_t b_bytes = static_cast<uint32_t>(p.n_pad) * 128;   // one K block of activations
  const uint32_t a_stage = C * kATileBytes, b_stage = C * b_bytes, raw_stage = C * kRawBytes;
  uint8_t* a_tiles = smem;                                     // [S][C][16 KB] decoded weights
  uint8_t* b_tiles = smem + static_cast<size_t>(S) * a_stage;  // [S][C][n_pad][128 B] activations
  uint8_t* raw = b_tiles + static_cast<size_t>(S) * b_stage;   // [R][C][kRawBytes]
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw + static_cast<size_t>(R) * raw_stage);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + kMaxRawStages;
  uint64_t* a_full = raw_empty + kMaxRawStages;
  uint64_t* b_full = a_full + kMaxOpStages;
  uint64_t* op_empty = b_full + kMaxOpStages;
  uint64_t* done = op_empty + kMaxOpStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int nt = blockIdx.x, j = blockIdx.y;
  const int kb0 = j * p.nkb_cta;
  const int nst = p.nkb_cta / C;   // stages to run
  const uint32_t ncols = pow2_at_least(static_cast<uint32_t>(p.n_pad), 32);
  const bool tl_on = p.tl != nullptr && tid == 0;
  __shared__ uint64_t tt[kTlStamps];   // timeline stamps (thread 0)
  if (tl_on)
    for (int i = 0; i < kTlStamps; ++i) tt[i] = 0;
  if (tl_on) tt[0] = global_ns();

  if (tid == 0) {
    s_abort = 0;
    s_raw_issued = 0;
    s_act_issued = 0;
    for (int i = 0; i < kMaxRawStages; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], kDecoderWarps);   // one arrival per decoder warp
    }
    for (int i = 0; i < kMaxOpStages; ++i) {
      mbar_init(&a_full[i], kDecoderWarps);
      mbar_init(&b_full[i], 1);
      mbar_init(&op_empty[i], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
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
  const uint32_t tmem = *tmem_slot;
  const bool geglu = p.out_geglu != nullptr;
  const float ds = geglu ? __fmul_rn(*p.sa, *p.sw) : 1.0f;
  const float rs = geglu ? (p.geglu_nvfp4 ? *p.sq : 1.0f / *p.sq) : 1.0f;   // four-bit: ts itself
  pdl_trigger();   // after TMEM is held (see the FP8 GEMM)

  if (tid == 0) {
    // ---------------- producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_a = l2_policy_evict_last();
    const uint8_t* wsrc = p.wpk + (static_cast<size_t>(nt) * p.nkb_total + kb0) * kRawBytes;
    const int pre = min(R, nst);
    for (int i = 0; i < pre; ++i) {
      mbar_arrive_expect_tx(&raw_full[i], raw_stage);
      bulk_load(raw + static_cast<size_t>(i) * raw_stage, wsrc + static_cast<size_t>(i) * raw_stage, raw_stage,
                &raw_full[i], pol_w);
    }
    int raw_issued = pre, act_issued = 0;
    pdl_wait();   // the activations are written by the previous kernel
    if (tl_on) tt[1] = global_ns();
    for (int st = 0; st < nst; ++st) {
      const int slot = st % S;
      if (st >= S && !mbar_wait(&op_empty[slot], static_cast<uint32_t>((st / S) - 1) & 1u)) {
        atomicOr(p.err, kErrPipelineTimeout);
        s_abort = 1;
        break;
      }
      mbar_arrive_expect_tx(&b_full[slot], b_stage);
      if (C == 1)   // a plain 2-D box when a stage holds one K block (the 3-D view measured slower)
        tma_load_2d(b_tiles + static_cast<size_t>(slot) * b_stage, &tmA, &b_full[slot], (kb0 + st) * kKb, 0, pol_a);
      else
        tma_load_3d(b_tiles + static_cast<size_t>(slot) * b_stage, &tmA, &b_full[slot], 0, 0, kb0 + st * C, pol_a);
      ++act_issued;
      const int ns = st + R;   // refill the raw slot stage st occupied
      if (ns < nst) {
        const int r = ns % R;
        if (!mbar_wait(&raw_empty[r], static_cast<uint32_t>((ns / R) - 1) & 1u)) {
          atomicOr(p.err, kErrPipelineTimeout);
          s_abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&raw_full[r], raw_stage);
        bulk_load(raw + static_cast<size_t>(r) * raw_stage, wsrc + static_cast<size_t>(ns) * raw_stage, raw_stage,
                  &raw_full[r], pol_w);
        ++raw_issued;
      }
    }
    s_raw_issued = raw_issued;
    s_act_issued = act_issued;
  } else if (tid == 32) {
    // ---------------- MMA issuer
    const uint32_t idesc = make_idesc_f16(kTileN, static_cast<uint32_t>(p.n_pad));
    for (int st = 0; st < nst; ++st) {
      const int slot = st % S;
      const uint32_t par = static_cast<uint32_t>(st / S) & 1u;
      if (!mbar_wait(&a_full[slot], par) || !mbar_wait(&b_full[slot], par)) {
        atomicOr(p.err, kErrPipelineTimeout);
        s_abort = 1;
        break;
      }
      tc_fence_after();
      for (int c = 0; c < C; ++c) {
        const uint32_t aa = smem_u32(a_tiles + static_cast<size_t>(slot) * a_stage + c * kATileBytes);
        const uint32_t ba = smem_u32(b_tiles + static_cast<size_t>(slot) * b_stage + c * b_bytes);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc_mma<false>(tmem, sw128_kmajor_desc(aa + k * 32), sw128_kmajor_desc(ba + k * 32), idesc,
                        (st > 0 || c > 0 || k > 0) ? 1u : 0u);
      }
      tc_commit(&op_empty[slot]);
    }
    tc_commit(done);
  } else if (warp >= 4) {
    // ---------------- decoders: kRowParts threads per weight row `row` of each block,
    // thread `part` expanding chunks part * kChunksPer .. + kChunksPer - 1 (elements
    // 8 per chunk) of that row
    const int row = (tid - 128) & 127;
    const int part = (tid - 128) >> 7;
    for (int st = 0; st < nst; ++st) {
      const int r = st % R;
      if (!mbar_wait(&raw_full[r], static_cast<uint32_t>(st / R) & 1u)) {
        atomicOr(p.err, kErrPipelineTimeout);
        s_abort = 1;
        break;
      }
      uint32_t codes[2][kChunksPer], sc[2];   // C <= 2: unrolled, so they stay in registers
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (c >= C) break;
        const uint8_t* src = raw + static_cast<size_t>(r) * raw_stage + c * kRawBytes;
        if constexpr (kChunksPer == 4) {
          const uint4 c0 = *reinterpret_cast<const uint4*>(src + row * 32 + part * 16);
          codes[c][0] = c0.x; codes[c][1] = c0.y; codes[c][2] = c0.z; codes[c][3] = c0.w;
        } else {
          const uint2 c0 = *reinterpret_cast<const uint2*>(src + row * 32 + part * 8);
          codes[c][0] = c0.x; codes[c][1] = c0.y;
        }
        sc[c] = *reinterpret_cast<const uint32_t*>(src + kCodeBytes + row * 4);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&raw_empty[r]);
      const int slot = st % S;
      if (st >= S && !mbar_wait(&op_empty[slot], static_cast<uint32_t>((st / S) - 1) & 1u)) {
        atomicOr(p.err, kErrPipelineTimeout);
        s_abort = 1;
        break;
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (c >= C) break;
        const uint32_t dst = smem_u32(a_tiles + static_cast<size_t>(slot) * a_stage + c * kATileBytes) + row * 128;
#pragma unroll
        for (int i = 0; i < kChunksPer; ++i) {   // 16-byte chunk q = elements 8q..8q+7, block scale q / 2
          const int q = part * kChunksPer + i;
          const __half bs = e4m3_half(static_cast<uint8_t>((sc[c] >> (8 * (q >> 1))) & 0xffu));
          st_shared_v4(dst + ((q ^ (row & 7)) << 4), decode8(codes[c][i], __half2(bs, bs)));
        }
      }
      fence_async_smem();   // generic-proxy writes -> tensor-core reads
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[slot]);
    }
  }

  // ---------------- epilogue: warps w, w + 4 and w + 8 share TMEM lane quarter w % 4 and
  // take every third 16-column chunk (activation rows)
  pdl_wait();   // the output buffers may still be read by earlier kernels until then
  if (!mbar_wait(done, 0)) {
    atomicOr(p.err, kErrPipelineTimeout);
    s_abort = 1;
  }
  if (tl_on) tt[2] = global_ns();
  tc_fence_after();
  __syncthreads();
  const bool abort = s_abort != 0;
  const int quarter = warp & 3, colset = warp >> 2;
  const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  const int n_local = quarter * 32 + lane;   // TMEM lane == weight row == output column in the tile
  __syncwarp();
  for (int c = colset * 16; c < p.n_pad; c += 16 * (kThreads / 128)) {
    float v[16];
    tmem_ld16(t_row + static_cast<uint32_t>(c), v);
    if (abort) continue;
    if (geglu) {
      // lanes 0-15 of a warp hold gate columns, lanes 16-31 the matching up columns, for 16
      // rows (the accumulator columns c .. c + 15)
      const size_t col = static_cast<size_t>(nt) * 64 + quarter * 16 + (lane & 15);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        // lanes 0-15 finish row c + i and lanes 16-31 row c + i + 8: each half passes the
        // other the value it lacks (the up value of row c + i, the gate value of row c + i + 8)
        const bool lo = lane < 16;
        const float got = __shfl_xor_sync(0xffffffffu, lo ? v[i + 8] : v[i], 16);
        const int m = c + i + (lo ? 0 : 8);
        const float x = (lo ? v[i] : got) * ds, u = (lo ? got : v[i + 8]) * ds;
        const float mv = 0.5f * x * (1.f + tanhf(0.7978845608028654f * fmaf(0.044715f * x, x * x, x))) * u;
        if (p.geglu_nvfp4) {
          // each half-warp holds one 16-column block of its row: its amax by shuffles
          // within the half
          float a = fabsf(mv);
          a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
          a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
          a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
          a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
          float den;
          const float bs = nvfp4_block(a, rs, &den);
          if (m < p.M)
            p.out_geglu[static_cast<size_t>(m) * (p.N / 2) + col] = nvfp4_one(mv, bs, den);
        } else if (m < p.M) {
          const uint8_t code = static_cast<uint8_t>(__nv_cvt_float_to_fp8(mv * rs, __NV_SATFINITE, __NV_E4M3));
          p.out_geglu[static_cast<size_t>(m) * (p.N / 2) + col] = e4m3_half(code);
        }
      }
    } else {
      float* plane = p.out + static_cast<size_t>(j) * p.M * p.N + static_cast<size_t>(nt) * kTileN + n_local;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (c + i < p.M) plane[static_cast<size_t>(c + i) * p.N] = v[i];
    }
  }

  if (tl_on) tt[3] = global_ns();
  // On an abandoned pipeline, let copies already in flight land before the CTA exits.
  if (abort && tid == 0) {
    const int ri = s_raw_issued, ai = s_act_issued;
    for (int r = 0; r < R && r < ri; ++r)
      mbar_wait(&raw_full[r], static_cast<uint32_t>((ri - 1 - r) / R) & 1u, 100000000ull);
    for (int slot = 0; slot < S && slot < ai; ++slot)
      mbar_wait(&b_full[slot], static_cast<uint32_t>((ai - 1 - slot) / S) & 1u, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (tl_on) {
    tt[4] = global_ns();
    tl_record(p.tl, kTlNvfp4, gridDim.y, blockIdx.y, tt);
  }
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// ---------------------------------------------------------------- packing

__global__ void tensor_scale_nvfp4_kernel(const unsigned* __restrict__ amax, float* __restrict__ ts) {
  const float a = __uint_as_float(*amax);
  *ts = a > 0.f ? a / 2688.0f : 1.0f;   // 2688 = 6 (E2M1 max) x 448 (E4M3 max)
}

// Packed row n of a gate|up weight (interleave): tile t = n / 128, 32-row group g,
// row w within it: w < 16 is gate row 64t + 16g + w, else up row F + 64t + 16g + w - 16,
// so lanes 0-15 and 16-31 of one epilogue warp hold matching gate/up columns.
__device__ __forceinline__ size_t source_row16(size_t n, int N, int interleave) {
  if (!interleave) return n;
  const size_t t = n / 128, g = (n % 128) / 32, w = n % 32;
  return w < 16 ? t * 64 + g * 16 + w : static_cast<size_t>(N / 2) + t * 64 + g * 16 + (w - 16);
}

// One thread per (row, 16-element block): block scale and eight code bytes.
__global__ void pack_nvfp4_kernel(const float* __restrict__ w, const float* __restrict__ gamma, int N, int K,
                                  const float* __restrict__ ts_ptr, uint8_t* __restrict__ out, int interleave) {
  const int nb = K / 16;
  const size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  if (idx >= static_cast<size_t>(N) * nb) return;
  const size_t n = idx / nb;
  const int b = static_cast<int>(idx % nb);
  const size_t src = source_row16(n, N, interleave);
  float wf[16];
  float amax_b = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int k = b * 16 + i;
    wf[i] = __fmul_rn(w[src * K + k], gamma ? gamma[k] : 1.0f);
    amax_b = fmaxf(amax_b, fabsf(wf[i]));
  }
  const float ts = *ts_ptr;
  const uint8_t bsc =
      static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fdiv_rn(amax_b, __fmul_rn(6.0f, ts)), __NV_SATFINITE, __NV_E4M3));
  const float den = __fmul_rn(__half2float(e4m3_half(bsc)), ts);
  alignas(8) uint8_t codes[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    codes[i] = den > 0.f ? static_cast<uint8_t>(__nv_cvt_float2_to_fp4x2(
                               make_float2(__fdiv_rn(wf[2 * i], den), __fdiv_rn(wf[2 * i + 1], den)), __NV_E2M1,
                               cudaRoundNearest))
                         : 0;
  const size_t nt = n / 128, r = n % 128;
  const int kb = b / 4, q = b % 4;
  uint8_t* blk = out + (nt * (K / kKb) + kb) * kRawBytes;
  *reinterpret_cast<uint2*>(blk + r * 32 + q * 8) = *reinterpret_cast<const uint2*>(codes);
  blk[kCodeBytes + r * 4 + q] = bsc;
}

}  // namespace

size_t nvfp4_packed_bytes(int N, int K) { return static_cast<size_t>(N / kTileN) * (K / kKb) * kRawBytes; }

cudaError_t pack_nvfp4(const float* w, const float* gamma, int N, int K, void* packed, float* ts_out,
                       unsigned* amax_scratch, cudaStream_t st, int geglu_interleave) {
  cudaError_t e = weight_amax_launch(w, gamma, N, K, amax_scratch, st);
  if (e != cudaSuccess) return e;
  tensor_scale_nvfp4_kernel<<<1, 1, 0, st>>>(amax_scratch, ts_out);
  const size_t n = static_cast<size_t>(N) * (K / 16);
  const int threads = 256;
  pack_nvfp4_kernel<<<static_cast<unsigned>((n + threads - 1) / threads), threads, 0, st>>>(
      w, gamma, N, K, ts_out, static_cast<uint8_t*>(packed), geglu_interleave);
  return cudaGetLastError();
}

int nvfp4_plan(int M, int N, int K, int s, Nvfp4Shape* g) {
  if (M < 1 || M > 256 || N <= 0 || K <= 0 || N % kTileN || K % 128) return FM_ERR_SHAPE;
  const int nkb_total = K / kKb;
  if (s < 1 || nkb_total % s) return FM_ERR_SHAPE;
  g->M = M;
  g->N = N;
  g->K = K;
  g->s = s;
  g->n_pad = (M + 15) / 16 * 16;
  g->nkb_total = nkb_total;
  g->nkb_cta = nkb_total / s;
  const size_t ctrl = align_up(kNumBars * 8 + 8, 256);
  // one K block per stage with the deepest operand ring that fits; two per stage
  // only if one would not leave room for two stages
  for (int chunk = 1; chunk <= 2; ++chunk) {
    if (g->nkb_cta % chunk) continue;
    const size_t stage = static_cast<size_t>(chunk) * (kATileBytes + static_cast<size_t>(g->n_pad) * 128);
    const size_t raw_stage = static_cast<size_t>(chunk) * kRawBytes;
    for (int raw = kMaxRawStages; raw >= 3; --raw) {
      const size_t fixed = raw * raw_stage + ctrl;
      if (fixed + 2 * stage > kSmemCap) continue;
      const int st = static_cast<int>(std::min<size_t>(kMaxOpStages, (kSmemCap - fixed) / stage));
      g->chunk = chunk;
      g->raw_stages = raw;
      g->op_stages = st;
      g->smem = 1024 + st * stage + fixed;
      return FM_OK;
    }
  }
  return FM_ERR_SHAPE;
}

bool nvfp4_tmap_act(CUtensorMap* map, const void* a, const Nvfp4Shape& g) {
  if (g.chunk == 1)
    return make_tmap_2d(map, a, 2, static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.M), kKb,
                        static_cast<uint32_t>(g.n_pad));
  return make_tmap_kblocks(map, a, 2, static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.M),
                           static_cast<uint32_t>(g.n_pad), static_cast<uint32_t>(g.chunk));
}

cudaError_t nvfp4_configure() {
  return configure_once(1, [] { return allow_max_dynamic_smem(reinterpret_cast<const void*>(nvfp4_gemm_kernel)); });
}

cudaError_t nvfp4_gemm_launch(const CUtensorMap& tmA, const void* wpk, const Nvfp4Shape& g, float* out,
                              __half* out_geglu, const float* sa, const float* sw, const float* sq, int* err,
                              const LaunchOpts& o, int geglu_nvfp4) {
  if (out_geglu && (g.s != 1 || !sa || !sw || !sq)) return cudaErrorInvalidValue;
  if (!out_geglu && !out) return cudaErrorInvalidValue;
  NvParams p;
  p.wpk = static_cast<const uint8_t*>(wpk);
  p.out = out;
  p.out_geglu = out_geglu;
  p.sa = sa;
  p.sw = sw;
  p.sq = sq;
  p.geglu_nvfp4 = geglu_nvfp4;
  p.tl = o.tl;
  p.M = g.M;
  p.N = g.N;
  p.nkb_total = g.nkb_total;
  p.nkb_cta = g.nkb_cta;
  p.n_pad = g.n_pad;
  p.op_stages = g.op_stages;
  p.raw_stages = g.raw_stages;
  p.chunk = g.chunk;
  p.err = err;
  LaunchOpts lo = o;
  lo.cluster = dim3(1, 1, 1);
  const dim3 grid(static_cast<unsigned>(g.N / kTileN), static_cast<unsigned>(g.s), 1);
  return launch(nvfp4_gemm_kernel, grid, dim3(kThreads), g.smem, lo, tmA, p);
}

}  // namespace fm
