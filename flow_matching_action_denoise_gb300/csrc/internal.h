// Declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "fmad.h"

namespace fm {

// Error-word bits set by kernels that abandon a bounded wait.
constexpr int kErrPipelineTimeout = 1;

// ---------------------------------------------------------------- launching
struct LaunchOpts {
  cudaStream_t stream = nullptr;
  bool pdl = false;      // Programmatic Dependent Launch attribute
  dim3 cluster{1, 1, 1};
  // Selective launch (standalone timing of one kernel of a sequence): when seq is set,
  // each launch takes the next index from *seq and only index `only` is issued.
  int* seq = nullptr;
  int only = -1;
  // Diagnostic timeline buffer (see tl_record in ptx.cuh); nullptr = off.
  unsigned long long* tl = nullptr;
};

template <typename... KArgs, typename... Args>
inline cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, const LaunchOpts& o,
                          Args&&... args) {
  if (o.seq) {
    const int idx = (*o.seq)++;
    if (o.only >= 0 && idx != o.only) return cudaSuccess;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = o.stream;
  cudaLaunchAttribute attrs[2];
  unsigned n = 0;
  if (o.pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (o.cluster.x * o.cluster.y * o.cluster.z > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = o.cluster.x;
    attrs[n].val.clusterDim.y = o.cluster.y;
    attrs[n].val.clusterDim.z = o.cluster.z;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Largest dynamic shared memory `kernel` may request on the current device (the
// opt-in per-block maximum minus the kernel's static shared memory); sets it.
cudaError_t allow_max_dynamic_smem(const void* kernel, size_t* granted = nullptr);
// Run a kernel family's one-time attribute setup (family 0..3) once per device.
cudaError_t configure_once(int family, cudaError_t (*fn)());

// ---------------------------------------------------------------- tensor maps
// 2-D tensor map over a row-major [outer][inner] array of 1- or 2-byte elements,
// 128-byte swizzle, zero fill out of bounds. Returns false on failure.
bool make_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner, uint64_t outer,
                  uint32_t box_inner, uint32_t box_outer);
// 3-D view of a row-major [rows][K] array as (128-byte K block inner, rows, K blocks):
// one box brings `blocks` consecutive K blocks of box_rows rows, laid out in shared
// memory as [blocks][box_rows][128 B] with the 128-byte swizzle.
bool make_tmap_kblocks(CUtensorMap* map, const void* base, int elem_bytes, uint64_t K, uint64_t rows,
                       uint32_t box_rows, uint32_t blocks);

// ---------------------------------------------------------------- skinny GEMM
struct GemmShape {
  int M, N, K;
  int fp8;        // 1: E4M3 operands, 0: BF16 operands
  int s;          // K-split
  int cs;         // cluster size reducing consecutive slices (divides s)
  int n_pad;      // MMA N (M rounded up to 16)
  int nkb_total;  // 128-byte K blocks
  int nkb_cta;    // K blocks per CTA
  int chunk;      // K blocks per pipeline stage (one weight copy + one activation box)
  int stages;     // pipeline stages in shared memory
  int tile;       // weight rows per CTA (MMA M): 128, or 64 (plain placement only)
  size_t smem;    // dynamic shared memory bytes
};
// Fills the derived fields; returns FM_OK or FM_ERR_SHAPE.
int gemm_plan(int M, int N, int K, int fp8, int s, int cs, GemmShape* g, int tile = 128);
// Activation tensor map: A [M][K] in K blocks of 128 bytes, box = chunk blocks x n_pad rows.
bool gemm_tmap_act(CUtensorMap* map, const void* a, const GemmShape& g);
// out: fp32 partial planes [s/cs][M][N]; or, with out_bf16 (requires cs == s), the
// dequantised product bf16(sum * fp32(*sa * *sw)) as [M][N].
// out_geglu (requires cs == s and a gate|up weight packed with interleave): the
// epilogue applies m = gelu_tanh(g) * u to the dequantised sums and writes Q(m, *sq)
// as [M][N/2] codes (E4M3 bytes if geglu_fp8, else bf16).
// wpk: packed weight tiles (1024-byte aligned, fm_pack_weight layout).
// Row work fused into a skinny GEMM. mode 1 (epilogue, requires cs == s): the gated
// residual x[m][n] += gate[n] * (sum * fp32(sa * sw)) on the finished sums, and
// ssq[n / 128][m] = that 128-column tile's sum of the new x^2 (no partial planes).
// mode 2 (prologue, the whole K range in the stages: gemm_mode2_ok): the activation
// operand is built from x [M][K] instead of loaded: Q(x * rsqrt(sum_t ssq[t][m] / K +
// eps) * (1 + scale) + shift), E4M3 with 1/sqa or bf16; the first n-tile's CTAs also
// store their K range of it in q_out [M][K].
struct GemmFuse {
  int mode = 0;
  float* x = nullptr;
  const float* gate = nullptr;
  float* ssq = nullptr;
  const float* scale = nullptr;
  const float* shift = nullptr;
  const float* sqa = nullptr;
  float eps = 0.f;
  void* q_out = nullptr;
};
bool gemm_mode2_ok(const GemmShape& g);
// out_qkv8 (requires cs == s): E4M3 codes of the dequantised product with the static
// scales s_qkv[0..2] for columns [0, nq), [nq, nq + nk), [nq + nk, N) (Q, K, V).
cudaError_t gemm_launch(const void* wpk, const CUtensorMap& tmA, const GemmShape& g, float* out, int* err,
                        const LaunchOpts& o, __nv_bfloat16* out_bf16 = nullptr, const float* sa = nullptr,
                        const float* sw = nullptr, void* out_geglu = nullptr, int geglu_fp8 = 0,
                        const float* sq = nullptr, uint8_t* out_qkv8 = nullptr, const float* s_qkv = nullptr,
                        int nq = 0, int nk = 0, const GemmFuse* fuse = nullptr,
                        const void* l2_prefetch = nullptr, size_t l2_prefetch_bytes = 0);
// l2_prefetch (16-byte aligned, bytes a multiple of 16): a range the kernel's CTAs
// prefetch into L2 once their own weight copies are issued, each its share (the next
// GEMM's weights, for CTAs of that GEMM that cannot be resident early).
cudaError_t gemm_configure();   // one-time function attributes (shared memory, clusters)

// ---------------------------------------------------------------- O GEMM + consumer
// The O projection with its consumer in the epilogue (ofuse.cu): one cluster spans the
// N / 128 <= 8 column tiles, each CTA the whole K of its 128 weight rows (E4M3 operands).
struct OConsumerShape {
  int M, N, K;
  int n_pad;   // MMA N (M rounded up to 16, <= 64)
  int nkb;     // 128-byte K blocks (all resident)
  int chunk;   // K blocks per TMA transaction
  size_t smem;
};
int o_consumer_plan(int M, int N, int K, OConsumerShape* g);
// Activation tensor map: A [M][K] E4M3 in K blocks, box = chunk blocks x n_pad rows.
bool o_consumer_tmap(CUtensorMap* map, const void* a, const OConsumerShape& g);
cudaError_t o_consumer_configure();
// x <- x + gate * (A W^T) * fp32(sa * sw); q = E4M3(AdaRMSNorm(x; scale, shift) * (1 / sq))
cudaError_t o_consumer_launch(const CUtensorMap& tmA, const void* wpk, const OConsumerShape& g, const float* sa,
                              const float* sw, const float* gate, float* x, const float* scale, const float* shift,
                              const float* sq, float eps, uint8_t* q, int* err, const LaunchOpts& o);

// ---------------------------------------------------------------- NVFP4-weight GEMM
struct Nvfp4Shape {
  int M, N, K;
  int s;           // K-split: partial planes [s][M][N]
  int n_pad;       // MMA N (M rounded up to 16)
  int nkb_total;   // 64-element K blocks
  int nkb_cta;
  int op_stages;   // decoded-operand pipeline stages
  int raw_stages;  // packed-weight ring stages
  int chunk;       // K blocks per stage
  size_t smem;
};
int nvfp4_plan(int M, int N, int K, int s, Nvfp4Shape* g);
// Activation tensor map: f16 values of E4M3 codes [M][K], box = 64 elements x n_pad rows.
bool nvfp4_tmap_act(CUtensorMap* map, const void* a, const Nvfp4Shape& g);
cudaError_t nvfp4_configure();
// out: fp32 partial planes [s][M][N]; or out_geglu (s == 1, gate|up packed with
// interleave): f16 values of E4M3(gelu(g) u * (1/s_q)) [M][N/2], g, u dequantised by fp32(sa * sw);
// with geglu_nvfp4 instead the four-bit activation values e * bs of gelu(g) u with tensor scale s_q.
cudaError_t nvfp4_gemm_launch(const CUtensorMap& tmA, const void* wpk, const Nvfp4Shape& g, float* out,
                              __half* out_geglu, const float* sa, const float* sw, const float* sq, int* err,
                              const LaunchOpts& o, int geglu_nvfp4 = 0);
size_t nvfp4_packed_bytes(int N, int K);
cudaError_t pack_nvfp4(const float* w, const float* gamma, int N, int K, void* packed, float* ts_out,
                       unsigned* amax_scratch, cudaStream_t st, int geglu_interleave);
// max |w[n][k] * gamma[k]| (fp32 products) as the bits of a non-negative float.
cudaError_t weight_amax_launch(const float* w, const float* gamma, int N, int K, unsigned* amax, cudaStream_t st);

// Packing
size_t packed_weight_bytes(int N, int K, int fmt);
// geglu_interleave: pack a gate|up weight [2F][K] so tile t holds, in alternate rows, gate row 64t+i and
// up row F+64t+i (i = 0..63)
cudaError_t pack_weight(const float* w, const float* gamma, int N, int K, int fmt, void* packed, float* scale_out,
                        unsigned* amax_scratch, cudaStream_t st, int geglu_interleave = 0);

// ---------------------------------------------------------------- row kernels
// Storage of a quantised GEMM operand (RowArgs::q_fp8, AttnArgs::out_fp8):
// 0 = bf16 values, 1 = E4M3 codes, 2 = E4M3 codes stored as their f16 values,
// 3 = four-bit (NVFP4) activations stored as the f16 values e * bs (quant.cuh).
constexpr int kQFp8AsF16 = 2;
constexpr int kQNvfp4AsF16 = 3;
// y[m][n] = bf16(sum_j planes[j][m][n] * fp32(sa * sw)) for s K-slice planes [s][M][N].
// With vt (nullable) the columns n >= nv0 (the values V) are also written transposed:
// vt[(n - nv0) * m_pad + m] (m_pad: M rounded up to 8), the chunk's V^T attention reads.
cudaError_t qkv_finalize_launch(const float* planes, int s, int M, int N, const float* sa, const float* sw,
                                __nv_bfloat16* out, __nv_bfloat16* vt, int nv0, int m_pad, const LaunchOpts& o);
struct RowArgs {
  int M, N;
  // residual update from GEMM partials: x += gate * (sum_p parts[p] * fp32(sa*sw) + bias)
  const float* parts;
  int nparts;
  const float* sa;
  const float* sw;
  const float* bias;
  const float* gate;
  float* x;
  const float* x_src;   // if non-null, x is first loaded from here (single-layer entry)
  // Euler tail: a += dt * (AdaRMSNorm_f(x) * gamma_f . w_out^T + b_out)
  int do_tail;
  const float* scale_f;
  const float* shift_f;
  const float* gamma_f;
  const __nv_bfloat16* w_out;
  const float* b_out;
  float* a;
  int A;
  float dt;
  // head: x = a . w_in^T + b_in
  int do_head;
  const __nv_bfloat16* w_in;
  const float* b_in;
  // AdaRMSNorm + quantise into q
  int do_quant;
  const float* scale;
  const float* shift;
  const float* sq;
  void* q;
  int q_fp8;
  float eps;
  // per-tile sums of squares for a following normalising GEMM prologue: the row's sum
  // of x^2 (after the head, if any) into ssq[0][m], zeros into ssq[1..ssq_tiles-1][m]
  float* ssq;
  int ssq_tiles;
  // decision timestamps (globaltimer ns): stamp_kind 1 = CTA 0 writes stamp[0] at its
  // start and clears stamp[1]; 2 = every CTA raises stamp[1] to its end time
  unsigned long long* stamp;
  int stamp_kind;
  unsigned long long* tl;   // diagnostic timeline (set from LaunchOpts by row_launch)
};
cudaError_t row_launch(const RowArgs& r, const LaunchOpts& o);
// Decision noise: out[i] (i < n) from Philox4x32-10 block i / 4 with counter
// (i / 4, 0, counter_lo, counter_hi) and key (seed_lo, seed_hi); words (w0, w1) give
// elements 4b, 4b+1 and (w2, w3) give 4b+2, 4b+3 by Box-Muller (in double, rounded to
// float). raw != nullptr also stores the four words of every block.
cudaError_t philox_noise_launch(float* out, int64_t n, uint64_t seed, uint64_t counter, uint32_t* raw,
                                cudaStream_t st);



struct AttnArgs {
  const __nv_bfloat16* qkv;     // [M][(H+2Hkv)*Dh] dequantised Q | K | V
  const __nv_bfloat16* kpre;    // [P][Hkv][Dh] of this layer
  const __nv_bfloat16* vtpre;   // [Hkv][Dh][p_pad] of this layer (values transposed)
  int p_pad;                    // P rounded up to a multiple of 8
  void* out;                    // [M][H*Dh] codes
  const float* s_out;
  int out_fp8;
  int M, P, H, Hkv;
  int kc;       // keys per slice (multiple of 64, <= 192)
  int nsplit;   // slices = cluster size (<= 8)
  int* err;
  // FP8 attention: qkv holds E4M3 codes [M][(H+2Hkv)*Dh] (bytes), the prefix comes
  // from its E4M3 copies, s_qkv points at the three static scales (Q, K, V)
  int fp8 = 0;
  const uint8_t* kpre8 = nullptr;    // [P][Hkv][Dh] of this layer
  const uint8_t* vtpre8 = nullptr;   // [Hkv][Dh][p16] of this layer
  int p16 = 0;                       // P rounded up to a multiple of 16
  const float* s_qkv = nullptr;
  // the chunk's values transposed [Hkv][Dh][m_pad] (bf16 attention; nullable: the wide
  // slice then gathers them from qkv)
  const __nv_bfloat16* vtc = nullptr;
  int m_pad = 0;
};
// Slice plan for P + M keys; FM_ERR_SHAPE when they need more than 8 x 192.
int attn_plan(int M, int P, int* kc, int* nsplit);
// attn_plan, then (bf16 attention on grids too large for the split head dims) the wide
// slice of 256 keys when its clusters need fewer waves of the GPU (device occupancy
// query; without a device the default plan). G: query heads per KV head.
int attn_plan_launch(int M, int P, int G, int Hkv, int fp8, int sms, int* kc, int* nsplit);
// Clusters of the attention kernel for (kc, nsplit, fp8, dv) resident at once; 0 when
// the query fails.
int attn_clusters_per_wave(int kc, int nsplit, int fp8, int dv);
size_t attn_smem_bytes(int kc, int nsplit, int fp8, int dv);   // dv: head dims of O per CTA
cudaError_t attn_launch(const AttnArgs& a, const LaunchOpts& o);
cudaError_t attn_configure();
// E4M3 copies of prefix rows [b, e) of every layer: k8 = E4M3(k * (1/s_k)), v8t likewise
// from the transposed bf16 values (row stride p16); s_k, s_v = ascale[l*8 + 5], [l*8 + 6].
cudaError_t prefix_quant_launch(const __nv_bfloat16* kcache, const __nv_bfloat16* vtcache, uint8_t* k8, uint8_t* v8t,
                                const float* ascale, int L, int P, int Hkv, int p_pad, int p16, int b, int e,
                                cudaStream_t st);
// v [L][rows][Hkv][Dh] -> vt[l][g][d][tok_begin + t] (row stride p_pad).
cudaError_t transpose_v_launch(const __nv_bfloat16* v, __nv_bfloat16* vt, int L, int rows, int Hkv, int p_pad,
                               int tok_begin, cudaStream_t st);

// ---------------------------------------------------------------- standalone GEMM + consumer
struct GemmConsumerArgs {
  const void* a;   // [M][K] fp8 codes or bf16
  int M, K, N, fmt, s;
  const void* w_packed;
  const float* s_a;
  const float* s_w;
  const float* bias;   // may be null
  float* x;            // [M][N] in/out
  const float* gate;
  const float* scale;
  const float* shift;
  float eps;
  const float* s_q;
  void* q;             // [M][N] codes
};
// Bytes of fp32 split-K partial planes the pair needs; FM_OK or a status.
int gemm_consumer_scratch_bytes(int M, int N, int K, int fmt, int s, size_t* bytes, const char** why);
// Validate, plan and launch the skinny GEMM into `scratch` (fp32 partial planes)
// and the fused consumer reading them. Returns FM_OK or a status; *why on failure.
int gemm_consumer_run(const GemmConsumerArgs& g, float* scratch, size_t scratch_bytes, int* err_word,
                      cudaStream_t st, const char** why);

// Device address of fm_gemm_consumer_noalloc's error word on device `dev` (nullptr
// before that entry point's first call there).
int* noalloc_error_word(int dev);

// Record `why` as the thread's last policy-free error (what fm_last_error(NULL)
// reports) and return `status`.
int record_error(int status, const char* why);

// ---------------------------------------------------------------- create-time kernels
// conds [S + (warm_t > 0)][d]: rows k < S for t_k = 1 - k/S (or the given vectors),
// row S for t = warm_t when warm_t > 0
cudaError_t cond_embed_launch(double* conds, int S, int d, const float* given, float warm_t, cudaStream_t st);
// One-step warm start input: a[m][j] = tau * noise[m][j] + (1 - tau) * prev[min(m + e, M - 1)][j]
cudaError_t warm_mix_launch(float* a, const float* prev, const float* noise, int M, int A, int e, float tau,
                            cudaStream_t st);
cudaError_t modtable_launch(const double* conds, int S, int d, const __nv_bfloat16* w_mod, const float* b_mod,
                            int nout, float* out, size_t out_step_stride, cudaStream_t st);
cudaError_t quant_e4m3_launch(const float* x, int64_t n, float scale, uint8_t* codes, cudaStream_t st);
cudaError_t scale_mul_launch(const float* a, const float* b, float* out, int n, cudaStream_t st);

}  // namespace fm
