// Policy object and C ABI of libfmad.so.
//
// A policy owns the plan of one decision - (L layers x 7 kernels) x S steps plus
// one step-head kernel - recorded once as a CUDA graph whose kernel nodes carry
// Programmatic Dependent Launch edges (news article "FlashRT-PAI", section "It
// optimises the relay": launch overlap; blog post "Embodied inference
// acceleration", section "CUDA Graph vs graph simplification": replay with the
// same parameters and addresses, new inputs written into agreed buffers).
// The caller's workspace is carved into named persistent buffers (the execution
// contract): packed weights and their scales, the static activation scales, the
// modulation table, the prefix KV cache, the noise/action buffer and the
// activation ping buffers. The execution-state capsule (snapshot / restore) is
// an in-process copy of the per-session regions, bound to the plan hash and the
// workspace address.

#include <cuda_bf16.h>

#include <algorithm>
#include <chrono>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "internal.h"

using fm::LaunchOpts;

namespace {

constexpr size_t kAlign = 1024;
constexpr uint64_t kCapsuleMagic = 0x3153504143444d46ull;   // "FMDCAPS1"

thread_local std::string g_last_error;

}  // namespace

// Device error word of the standalone building-block entry points (the policy
// keeps its own in its workspace).
__device__ int fm_standalone_err;

namespace {

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t total = 0;
  // [0, shared_end): read-only after create (packed weights, scales, modulation, the
  // in/out projections), shared by the policy's sessions; the rest is per-session state
  size_t shared_end = 0;
  std::vector<size_t> wpk;   // [L*4] packed weights
  size_t wscale, ascale, mod, modf, w_in, b_in, w_out, b_out, gamma_f, kcache, vcache, a, x, q, o, q2, mc;
  size_t vtc;    // NVFP4: the chunk's values transposed [Hkv][Dh][M rounded up to 8] (bf16)
  size_t qkvb;   // bf16 Q | K | V the attention reads (== y[0] unless NVFP4 reduces planes separately;
                 // E4M3 codes with FP8 attention)
  size_t kcache8, vcache8;   // FP8 attention: E4M3 copies of the prefix cache
  size_t kv8_bytes, v8_bytes, ascale_bytes;
  size_t ssq;   // [d/128][M] per-tile sums of squares of x (consumers inside the GEMMs)
  size_t stamps;   // [2] u64: globaltimer ns at the decision's first kernel start, last kernel end
  size_t prev;     // [M][A] fp32: the previous chunk, shifted by a warm start
  size_t y[4];
  size_t err, amax, conds;
  size_t kv_bytes, a_bytes, scale_bytes;
  size_t take(size_t bytes) {
    const size_t off = total;
    total = align_up(total + std::max<size_t>(bytes, 1));
    return off;
  }
};

struct Derived {
  int nqkv;
  int act_bytes;
  int fp8;
  int nvfp4;
  int q_store;   // quantised operand storage: 0 bf16, 1 E4M3 codes, 2 E4M3 codes as f16 values,
                 // 3 four-bit activation values e * bs as f16
  int act4;      // four-bit (NVFP4) activations: block scales from the activation, static tensor scale
  int attn_fp8;  // attention on E4M3 Q, K, V and probabilities
  // FP8/BF16: the consumers run inside the GEMMs - the O and down GEMM epilogues apply
  // the gated residual and emit per-tile sums of squares, the QKV and gate|up GEMMs
  // build their normalised, quantised operand in a prologue (5 kernels per layer)
  int rowfuse;
  // FM_FLAG_O_CONSUMER_IN_GEMM (FP8, d <= 1024, H * Dh <= 1024, M <= 64): the O GEMM and
  // its consumer in one kernel (ofuse.cu), 6 kernels per layer
  int ofuse;
  fm::OConsumerShape os;
  fm::GemmShape gs[4];
  fm::Nvfp4Shape ns[4];
  int gN[4], gK[4];
  int attn_kc, attn_nsplit;
  // fp32 partial planes GEMM g writes (its K-slices not reduced in the GEMM itself)
  int nparts(int g) const {
    return nvfp4 ? ns[g].s : ((rowfuse && (g == 1 || g == 3)) || (ofuse && g == 1)) ? 0 : gs[g].s / gs[g].cs;
  }
  int kernels_per_layer() const { return nvfp4 ? 8 : rowfuse ? 5 : ofuse ? 6 : 7; }
};

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
      n = 148;
  }
  return n;
}

int auto_split(int tiles, int nkb) {
  const int target = num_sms() * 3 / 4;
  for (int s = 1; s <= nkb; ++s)
    if (nkb % s == 0 && tiles * s >= target) return s;
  return nkb;
}

// auto_split for a GEMM whose CTAs take a whole SM (the NVFP4 kernel's shared memory):
// the grid is kept to one wave, the largest such split when auto_split's would spill
// over (measured: the W4A8 QKV GEMM at split 8, 160 CTAs, took two waves, 13.7 us per
// layer-step; at split 4, 80 CTAs, 9.4 us).
int auto_split_one_wave(int tiles, int nkb) {
  int s = auto_split(tiles, nkb);
  while (s > 1 && tiles * s > num_sms()) {
    --s;
    while (s > 1 && nkb % s) --s;
  }
  return s;
}

int cluster_for(int s) {
  int c = 8;
  while (c > 1 && s % c) c >>= 1;
  return c;
}

int validate(const fm_config* c, std::string* why) {
  if (!c) {
    *why = "config is NULL";
    return FM_ERR_INVALID_ARG;
  }
  if (c->abi_version != FM_ABI_VERSION) {
    *why = "abi_version mismatch";
    return FM_ERR_INVALID_ARG;
  }
  const bool fmt_ok = (c->weight_fmt == FM_FMT_FP8 && c->act_fmt == FM_FMT_FP8) ||
                      (c->weight_fmt == FM_FMT_BF16 && c->act_fmt == FM_FMT_BF16) ||
                      (c->weight_fmt == FM_FMT_NVFP4 && (c->act_fmt == FM_FMT_FP8 || c->act_fmt == FM_FMT_NVFP4));
  if (!fmt_ok) {
    *why = "unsupported weight/activation format pair";
    return FM_ERR_INVALID_ARG;
  }
  if (c->attn_fmt != FM_FMT_BF16 && c->attn_fmt != FM_FMT_FP8) {
    *why = "attn_fmt must be FM_FMT_BF16 or FM_FMT_FP8";
    return FM_ERR_INVALID_ARG;
  }
  if (c->attn_fmt == FM_FMT_FP8 && (c->weight_fmt != FM_FMT_FP8 || c->act_fmt != FM_FMT_FP8)) {
    *why = "FP8 attention is built for FP8 weights and activations";
    return FM_ERR_UNSUPPORTED;
  }
  if (c->cond_mode != FM_COND_TIME && c->cond_mode != FM_COND_GIVEN) {
    *why = "bad cond_mode";
    return FM_ERR_INVALID_ARG;
  }
  if (c->L < 1 || c->S < 1 || c->M < 1 || c->M > 256 || c->A < 1 || c->A > 32 || c->P < 0 || c->Dh != 128 ||
      c->H < 1 || c->Hkv < 1 || c->H % c->Hkv || c->d % 128 || c->d <= 0 || c->F % 128 || c->F <= 0 ||
      c->d > 12288) {
    *why = "shape precondition violated (d, F multiples of 128, d <= 12288, Dh == 128, H % Hkv == 0, "
           "1 <= M <= 256, 1 <= A <= 32)";
    return FM_ERR_SHAPE;
  }
  if (!(c->rms_eps > 0.f)) {
    *why = "rms_eps must be positive";
    return FM_ERR_INVALID_ARG;
  }
  if (!(c->warm_t >= 0.f && c->warm_t <= 1.f) || (c->warm_t > 0.f && c->cond_mode != FM_COND_TIME)) {
    *why = "warm_t must lie in [0, 1], and a warm start needs time conditioning";
    return FM_ERR_INVALID_ARG;
  }
  return FM_OK;
}

int derive(const fm_config* c, Derived* dv, std::string* why) {
  dv->nqkv = (c->H + 2 * c->Hkv) * c->Dh;
  dv->fp8 = c->act_fmt == FM_FMT_FP8;
  dv->nvfp4 = c->weight_fmt == FM_FMT_NVFP4;
  dv->act4 = c->act_fmt == FM_FMT_NVFP4;
  dv->q_store = dv->nvfp4 ? (dv->act4 ? fm::kQNvfp4AsF16 : fm::kQFp8AsF16) : dv->fp8;
  dv->attn_fp8 = c->attn_fmt == FM_FMT_FP8;
  dv->rowfuse = 0;
  dv->ofuse = 0;
  dv->act_bytes = dv->q_store == 1 ? 1 : 2;
  const int N[4] = {dv->nqkv, c->d, 2 * c->F, c->d};
  const int K[4] = {c->d, c->H * c->Dh, c->d, c->F};
  if (dv->nvfp4) {
    // NVFP4 weights: the GEMMs write fp32 partial planes (QKV's are reduced by a
    // separate kernel into bf16); the gate|up GEMM applies GeGLU itself, so it keeps
    // the whole K in one CTA.
    for (int g = 0; g < 4; ++g) {
      dv->gN[g] = N[g];
      dv->gK[g] = K[g];
      const int nkb = K[g] / 64;
      int s = c->ksplit[g] > 0 ? c->ksplit[g] : (g == 2 ? 1 : auto_split_one_wave(N[g] / 128, nkb));
      if (g == 2 && s != 1) {
        *why = "with NVFP4 weights the gate|up GEMM cannot be K-split (its epilogue applies GeGLU)";
        return FM_ERR_SHAPE;
      }
      if (fm::nvfp4_plan(c->M, N[g], K[g], s, &dv->ns[g]) != FM_OK) {
        char buf[160];
        snprintf(buf, sizeof buf, "NVFP4 GEMM %d: split %d does not divide %d K-blocks (N=%d, K=%d)", g, s, nkb,
                 N[g], K[g]);
        *why = buf;
        return FM_ERR_SHAPE;
      }
      memset(&dv->gs[g], 0, sizeof(fm::GemmShape));
    }
    if (fm::attn_plan_launch(c->M, c->P, c->H / c->Hkv, c->Hkv, dv->attn_fp8, num_sms(), &dv->attn_kc,
                             &dv->attn_nsplit) != FM_OK) {
      *why = "P + M keys exceed the attention plan's 8 slices x 192 keys";
      return FM_ERR_SHAPE;
    }
    return FM_OK;
  }
  memset(dv->ns, 0, sizeof dv->ns);
  for (int g = 0; g < 4; ++g) {
    dv->gN[g] = N[g];
    dv->gK[g] = K[g];
    const int nkb = K[g] * dv->act_bytes / 128;
    int s = c->ksplit[g] > 0 ? c->ksplit[g] : auto_split(N[g] / 128, nkb);
    // The QKV and gate|up GEMMs reduce all their K-slices inside one cluster (their
    // epilogues emit bf16 Q|K|V and the GeGLU output), so their split is 1, 2, 4 or 8.
    const bool whole_cluster = g == 0 || g == 2;
    if (whole_cluster && c->ksplit[g] <= 0)
      while (s > 8 || (s & (s - 1)) || nkb % s) --s;
    if (whole_cluster && (s > 8 || (s & (s - 1)))) {
      *why = "the QKV and gate|up K-splits must be 1, 2, 4 or 8 (their slices are reduced within one cluster)";
      return FM_ERR_SHAPE;
    }
    const int st = fm::gemm_plan(c->M, N[g], K[g], dv->fp8, s, cluster_for(s), &dv->gs[g]);
    if (st != FM_OK) {
      char buf[160];
      snprintf(buf, sizeof buf, "GEMM %d: split %d does not divide %d K-blocks (N=%d, K=%d)", g, s, nkb, N[g], K[g]);
      *why = buf;
      return st;
    }
  }
  if (fm::attn_plan_launch(c->M, c->P, c->H / c->Hkv, c->Hkv, dv->attn_fp8, num_sms(), &dv->attn_kc,
                           &dv->attn_nsplit) != FM_OK) {
    *why = "P + M keys exceed the attention plan's 8 slices x 192 keys";
    return FM_ERR_SHAPE;
  }
  // Consumers inside the GEMMs: the O and down GEMMs must finish every K slice in one
  // cluster (split = cluster <= 8) and the QKV and gate|up GEMMs must hold their whole
  // K range in shared memory; automatic splits are adjusted to get there.
  if (c->flags & FM_FLAG_FUSED_CONSUMERS) {
    fm::GemmShape cand[4] = {dv->gs[0], dv->gs[1], dv->gs[2], dv->gs[3]};
    bool ok = true;
    for (int g = 0; g < 4 && ok; ++g) {
      const int nkb = K[g] * dv->act_bytes / 128;
      int s = cand[g].s;
      if (g == 1 || g == 3) {
        if (c->ksplit[g] <= 0)
          while (s > 8 || (s & (s - 1)) || nkb % s) --s;
        ok = s == cluster_for(s) && s <= 8 &&
             fm::gemm_plan(c->M, N[g], K[g], dv->fp8, s, cluster_for(s), &cand[g]) == FM_OK;
      } else {
        while (!fm::gemm_mode2_ok(cand[g]) && c->ksplit[g] <= 0 && s * 2 <= 8 && nkb % (s * 2) == 0) {
          s *= 2;
          if (fm::gemm_plan(c->M, N[g], K[g], dv->fp8, s, cluster_for(s), &cand[g]) != FM_OK) break;
        }
        ok = fm::gemm_mode2_ok(cand[g]);
      }
    }
    if (ok) {
      for (int g = 0; g < 4; ++g) dv->gs[g] = cand[g];
      dv->rowfuse = 1;
    }
  }
  // The gate|up GEMM (N = 2F, the largest) in 64-row weight tiles when the doubled grid
  // still fits in one wave at two CTAs per SM: half the split-K partial bytes per CTA
  // (measured: expert_fp8_m50 5.74 -> 5.71 ms; with bf16 operands the CTAs need more
  // than half an SM's shared memory and it is not taken).
  if (!dv->rowfuse && dv->fp8 && (c->flags & FM_FLAG_O_CONSUMER_IN_GEMM) &&
      fm::o_consumer_plan(c->M, N[1], K[1], &dv->os) == FM_OK)
    dv->ofuse = 1;
  if (!dv->rowfuse) {   // (the consumers-inside-GEMMs placement keeps 128-row tiles)
    fm::GemmShape g64;
    const fm::GemmShape& g2 = dv->gs[2];
    if (fm::gemm_plan(c->M, N[2], K[2], dv->fp8, g2.s, g2.cs, &g64, 64) == FM_OK && g64.smem <= 113 * 1024 &&
        (N[2] / 64) * g2.s <= 2 * num_sms())
      dv->gs[2] = g64;
  }
  return FM_OK;
}

Layout make_layout(const fm_config* c, const Derived& dv) {
  Layout ly;
  const int L = c->L, d = c->d, S = c->S, M = c->M;
  const int wfmt = c->weight_fmt;
  ly.wpk.resize(static_cast<size_t>(L) * 4);
  for (int l = 0; l < L; ++l)
    for (int g = 0; g < 4; ++g) ly.wpk[l * 4 + g] = ly.take(fm::packed_weight_bytes(dv.gN[g], dv.gK[g], wfmt));
  ly.scale_bytes = static_cast<size_t>(L) * 4 * sizeof(float);
  ly.ascale_bytes = static_cast<size_t>(L) * 8 * sizeof(float);   // [L][8]: FM_SITE_* columns
  ly.wscale = ly.take(ly.scale_bytes);
  const int rows = S + (c->warm_t > 0.f ? 1 : 0);   // row S: the warm start's flow time
  ly.mod = ly.take(static_cast<size_t>(rows) * L * 6 * d * sizeof(float));
  ly.modf = ly.take(static_cast<size_t>(rows) * 2 * d * sizeof(float));
  ly.w_in = ly.take(static_cast<size_t>(d) * c->A * 2);
  ly.b_in = ly.take(static_cast<size_t>(d) * 4);
  ly.w_out = ly.take(static_cast<size_t>(d) * c->A * 2);
  ly.b_out = ly.take(static_cast<size_t>(c->A) * 4);
  ly.gamma_f = ly.take(static_cast<size_t>(d) * 4);
  ly.conds = ly.take(static_cast<size_t>(rows) * d * sizeof(double));
  ly.amax = ly.take(64);
  ly.shared_end = ly.total;
  // ---- per-session state
  ly.ascale = ly.take(ly.ascale_bytes);
  // K [L][P][Hkv][Dh]; V stored transposed [L][Hkv][Dh][P_pad], P_pad = P rounded up to 8
  ly.kv_bytes = static_cast<size_t>(L) * ((c->P + 7) / 8 * 8) * c->Hkv * c->Dh * 2;
  ly.kcache = ly.take(ly.kv_bytes);
  ly.vcache = ly.take(ly.kv_bytes);
  ly.a_bytes = static_cast<size_t>(M) * c->A * 4;
  ly.a = ly.take(ly.a_bytes);
  ly.x = ly.take(static_cast<size_t>(M) * d * 4);
  ly.q = ly.take(static_cast<size_t>(M) * d * dv.act_bytes);
  ly.o = ly.take(static_cast<size_t>(M) * c->H * c->Dh * dv.act_bytes);
  ly.q2 = ly.take(static_cast<size_t>(M) * d * dv.act_bytes);
  ly.mc = ly.take(static_cast<size_t>(M) * c->F * dv.act_bytes);
  for (int g = 0; g < 4; ++g)
    ly.y[g] = ly.take(g == 2 ? 0 :   // the gate|up GEMM writes the GeGLU output directly
                      (g == 0 && !dv.nvfp4) ? static_cast<size_t>(M) * dv.gN[0] * 2   // dequantised bf16 Q|K|V
                                            : static_cast<size_t>(dv.nparts(g)) * M * dv.gN[g] * 4);
  ly.qkvb = dv.nvfp4 ? ly.take(static_cast<size_t>(M) * dv.gN[0] * 2) : ly.y[0];
  ly.vtc = dv.nvfp4 ? ly.take(static_cast<size_t>(c->Hkv) * c->Dh * ((M + 7) / 8 * 8) * 2) : 0;
  ly.kv8_bytes = dv.attn_fp8 ? static_cast<size_t>(L) * c->P * c->Hkv * c->Dh : 0;
  ly.v8_bytes = dv.attn_fp8 ? static_cast<size_t>(L) * c->Hkv * c->Dh * ((c->P + 15) / 16 * 16) : 0;
  ly.kcache8 = ly.take(ly.kv8_bytes);
  ly.vcache8 = ly.take(ly.v8_bytes);
  ly.err = ly.take(64);
  ly.ssq = ly.take(static_cast<size_t>(c->d / 128) * M * sizeof(float));
  ly.stamps = ly.take(64);
  ly.prev = ly.take(ly.a_bytes);   // the chunk a warm start shifts
  return ly;
}

uint64_t fnv(uint64_t h, const void* p, size_t n) {
  const unsigned char* b = static_cast<const unsigned char*>(p);
  for (size_t i = 0; i < n; ++i) {
    h ^= b[i];
    h *= 1099511628211ull;
  }
  return h;
}

struct CapsuleHeader {
  uint64_t magic;
  uint32_t abi, header_bytes;
  uint64_t plan_hash;
  uint64_t ws_base;
  uint64_t kv_bytes, a_bytes, scale_bytes;
  int32_t L, P, Hkv, Dh, M, A;
  uint64_t decisions;
  uint8_t pad[256 - 8 - 8 - 8 - 8 - 24 - 24 - 8];
};
static_assert(sizeof(CapsuleHeader) == 256, "capsule header is 256 bytes");

}  // namespace

struct fm_policy {
  fm_config cfg;
  Derived dv;
  Layout ly;
  uint8_t* ws = nullptr;       // this policy's (or session's) workspace: capsules bind to it
  size_t ws_bytes = 0;
  uint8_t* shared = nullptr;   // layout offsets [0, shared_end): the base policy's workspace
  uint8_t* state = nullptr;    // layout offsets [shared_end, total)
  fm_policy* base = nullptr;   // a session's base policy (shares its weights)
  int sessions = 0;            // live sessions of this base policy
  CUtensorMap tmA[4];
  CUtensorMap tmO;   // the attention output as the fused O GEMM + consumer reads it
  cudaStream_t cap_stream = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaGraph_t warm_graph = nullptr;     // the one-step warm start (cfg.warm_t > 0)
  cudaGraphExec_t warm_exec = nullptr;
  bool have_prev = false;               // the noise/action buffer holds a decided chunk
  uint64_t plan_hash = 0;
  uint64_t decisions = 0;
  uint64_t host_submit_ns = 0;   // steady clock when the last decision was enqueued
  std::string err;
  CapsuleHeader hdr;   // staging for device-side snapshots (must outlive the async copy)

  template <typename T>
  T* at(size_t off) const {
    return reinterpret_cast<T*>(off < ly.shared_end ? shared + off : state + (off - ly.shared_end));
  }
  float* mod(int k, int l, int i) const {
    return at<float>(ly.mod) + ((static_cast<size_t>(k) * cfg.L + l) * 6 + i) * cfg.d;
  }
  float* modf(int k, int i) const { return at<float>(ly.modf) + (static_cast<size_t>(k) * 2 + i) * cfg.d; }
  float* wscale(int l, int g) const { return at<float>(ly.wscale) + l * 4 + g; }
  float* ascale(int l, int i) const { return at<float>(ly.ascale) + l * 8 + i; }
  int* errw() const { return at<int>(ly.err); }
};

namespace {

int fail(fm_policy* p, int status, const std::string& why) {
  if (p)
    p->err = why;
  else
    g_last_error = why;
  return status;
}

int cuda_fail(fm_policy* p, cudaError_t e, const char* where) {
  std::string s = std::string(where) + ": " + cudaGetErrorString(e);
  return fail(p, FM_ERR_CUDA, s);
}

#define FM_CUDA(p, call)                                       \
  do {                                                         \
    cudaError_t e_ = (call);                                   \
    if (e_ != cudaSuccess) return cuda_fail((p), e_, #call);   \
  } while (0)

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

// The device scale table [L][8] from the caller's [L][4] ([L][7] with FP8 attention).
std::vector<float> scale_table(const fm_config& c, const Derived& dv, const float* act_scales) {
  std::vector<float> sc(static_cast<size_t>(c.L) * 8, 1.0f);
  const int cols = dv.attn_fp8 ? 7 : 4;
  if ((dv.fp8 || dv.act4) && act_scales)
    for (int l = 0; l < c.L; ++l)
      for (int i = 0; i < cols; ++i) sc[static_cast<size_t>(l) * 8 + i] = act_scales[static_cast<size_t>(l) * cols + i];
  return sc;
}

// ---------------------------------------------------------------- tracing
// Optional recorder: after a kernel, copy the buffer it wrote into the trace.
struct Trace {
  uint8_t* base = nullptr;
  size_t off = 0;
  cudaStream_t st = nullptr;
  cudaError_t rec(const void* src, size_t bytes) {
    if (!base) return cudaSuccess;
    const cudaError_t e = cudaMemcpyAsync(base + off, src, bytes, cudaMemcpyDeviceToDevice, st);
    off += bytes;
    return e;
  }
};

// ---------------------------------------------------------------- the plan
// Kernels of layer l at step k. tail: -1 = next layer's norm (layer (l+1) mod L),
// otherwise the last layer of a decision step (Euler tail; head of step tail
// if tail < S).
// E4M3 copies of prefix rows [b, e) of every layer (FP8 attention), quantised with
// the layer's static K and V scales.
cudaError_t requant_prefix(fm_policy* p, int b, int e, cudaStream_t s) {
  const fm_config& c = p->cfg;
  return fm::prefix_quant_launch(p->at<__nv_bfloat16>(p->ly.kcache), p->at<__nv_bfloat16>(p->ly.vcache),
                                 p->at<uint8_t>(p->ly.kcache8), p->at<uint8_t>(p->ly.vcache8),
                                 p->at<float>(p->ly.ascale), c.L, c.P, c.Hkv, (c.P + 7) / 8 * 8,
                                 (c.P + 15) / 16 * 16, b, e, s);
}

cudaError_t enqueue_layer(fm_policy* p, int l, int k, bool step_end, const LaunchOpts& o, Trace* tr = nullptr) {
  const fm_config& c = p->cfg;
  const Derived& dv = p->dv;
  cudaError_t e;
  int* err = p->errw();
  float* y[4];
  size_t ybytes[4];
  for (int g = 0; g < 4; ++g) {
    y[g] = p->at<float>(p->ly.y[g]);
    ybytes[g] = g == 0 ? static_cast<size_t>(c.M) * dv.gN[0] * 2 : static_cast<size_t>(dv.nparts(g)) * c.M * dv.gN[g] * 4;
  }
  const int fp8 = dv.q_store;
  __nv_bfloat16* qkvb = p->at<__nv_bfloat16>(p->ly.qkvb);
  const size_t xbytes = static_cast<size_t>(c.M) * c.d * 4;
  const size_t ab = dv.act_bytes;
  Trace none;
  Trace& t = tr ? *tr : none;
#define FM_REC(ptr, bytes)                 \
  do {                                     \
    e = t.rec((ptr), (bytes));             \
    if (e != cudaSuccess) return e;        \
  } while (0)
  FM_REC(p->at<void>(p->ly.x), xbytes);
  if (!dv.rowfuse) FM_REC(p->at<void>(p->ly.q), static_cast<size_t>(c.M) * c.d * ab);
  float* ssq = p->at<float>(p->ly.ssq);
  // consumers inside the GEMMs: the QKV GEMM normalises and quantises x itself
  fm::GemmFuse fq;
  fq.mode = 2;
  fq.x = p->at<float>(p->ly.x);
  fq.ssq = ssq;
  fq.scale = p->mod(k, l, 0);
  fq.shift = p->mod(k, l, 1);
  fq.sqa = p->ascale(l, FM_SITE_ATTN_IN);
  fq.eps = c.rms_eps;
  fq.q_out = p->at<void>(p->ly.q);
  const fm::GemmFuse* fqp = dv.rowfuse ? &fq : nullptr;

  // QKV: the epilogue dequantises and rounds to bf16, the operand attention reads
  // (NVFP4: partial planes, reduced and rounded by a separate kernel)
  if (dv.nvfp4) {
    e = fm::nvfp4_gemm_launch(p->tmA[0], p->at<void>(p->ly.wpk[l * 4 + 0]), dv.ns[0], y[0], nullptr, nullptr, nullptr,
                              nullptr, err, o);
    if (e != cudaSuccess) return e;
    e = fm::qkv_finalize_launch(y[0], dv.ns[0].s, c.M, dv.gN[0], p->ascale(l, FM_SITE_ATTN_IN), p->wscale(l, 0), qkvb,
                                p->at<__nv_bfloat16>(p->ly.vtc), (c.H + c.Hkv) * c.Dh, (c.M + 7) / 8 * 8, o);
  } else if (dv.attn_fp8) {   // E4M3 Q | K | V codes with their static scales
    e = fm::gemm_launch(p->at<void>(p->ly.wpk[l * 4 + 0]), p->tmA[0], dv.gs[0], nullptr, err, o, nullptr,
                        p->ascale(l, FM_SITE_ATTN_IN), p->wscale(l, 0), nullptr, 0, nullptr,
                        reinterpret_cast<uint8_t*>(qkvb), p->ascale(l, FM_SITE_Q), c.H * c.Dh, c.Hkv * c.Dh, fqp);
  } else {
    e = fm::gemm_launch(p->at<void>(p->ly.wpk[l * 4 + 0]), p->tmA[0], dv.gs[0], nullptr, err, o, qkvb,
                        p->ascale(l, FM_SITE_ATTN_IN), p->wscale(l, 0), nullptr, 0, nullptr, nullptr, nullptr, 0, 0,
                        fqp);
  }
  if (e != cudaSuccess) return e;
  if (dv.rowfuse) FM_REC(p->at<void>(p->ly.q), static_cast<size_t>(c.M) * c.d * ab);
  FM_REC(qkvb, dv.attn_fp8 ? ybytes[0] / 2 : ybytes[0]);

  fm::AttnArgs at;
  at.qkv = qkvb;
  const int p_pad = (c.P + 7) / 8 * 8;
  at.kpre = p->at<__nv_bfloat16>(p->ly.kcache) + static_cast<size_t>(l) * c.P * c.Hkv * c.Dh;
  at.vtpre = p->at<__nv_bfloat16>(p->ly.vcache) + static_cast<size_t>(l) * c.Hkv * c.Dh * p_pad;
  at.p_pad = p_pad;
  at.err = err;
  at.out = p->at<void>(p->ly.o);
  at.s_out = p->ascale(l, FM_SITE_ATTN_OUT);
  at.out_fp8 = fp8;
  at.M = c.M;
  at.P = c.P;
  at.H = c.H;
  at.Hkv = c.Hkv;
  at.kc = dv.attn_kc;
  at.nsplit = dv.attn_nsplit;
  if (dv.nvfp4) {
    at.vtc = p->at<__nv_bfloat16>(p->ly.vtc);
    at.m_pad = (c.M + 7) / 8 * 8;
  }
  if (dv.attn_fp8) {
    const int p16 = (c.P + 15) / 16 * 16;
    at.fp8 = 1;
    at.kpre8 = p->at<uint8_t>(p->ly.kcache8) + static_cast<size_t>(l) * c.P * c.Hkv * c.Dh;
    at.vtpre8 = p->at<uint8_t>(p->ly.vcache8) + static_cast<size_t>(l) * c.Hkv * c.Dh * p16;
    at.p16 = p16;
    at.s_qkv = p->ascale(l, FM_SITE_Q);
  }
  e = fm::attn_launch(at, o);
  if (e != cudaSuccess) return e;
  FM_REC(p->at<void>(p->ly.o), static_cast<size_t>(c.M) * c.H * c.Dh * ab);

  // consumers inside the GEMMs: the O GEMM applies the gated residual itself
  fm::GemmFuse fo;
  fo.mode = 1;
  fo.x = p->at<float>(p->ly.x);
  fo.gate = p->mod(k, l, 2);
  fo.ssq = ssq;
  if (dv.nvfp4)
    e = fm::nvfp4_gemm_launch(p->tmA[1], p->at<void>(p->ly.wpk[l * 4 + 1]), dv.ns[1], y[1], nullptr, nullptr, nullptr,
                              nullptr, err, o);
  else if (dv.ofuse)   // the O GEMM with its consumer: x and the pre-MLP operand q2 (no row kernel)
    e = fm::o_consumer_launch(p->tmO, p->at<void>(p->ly.wpk[l * 4 + 1]), dv.os, p->ascale(l, FM_SITE_ATTN_OUT),
                              p->wscale(l, 1), p->mod(k, l, 2), p->at<float>(p->ly.x), p->mod(k, l, 3),
                              p->mod(k, l, 4), p->ascale(l, FM_SITE_MLP_IN), c.rms_eps, p->at<uint8_t>(p->ly.q2), err,
                              o);
  else if (dv.rowfuse)
    e = fm::gemm_launch(p->at<void>(p->ly.wpk[l * 4 + 1]), p->tmA[1], dv.gs[1], nullptr, err, o, nullptr,
                        p->ascale(l, FM_SITE_ATTN_OUT), p->wscale(l, 1), nullptr, 0, nullptr, nullptr, nullptr, 0, 0,
                        &fo);
  else
    e = fm::gemm_launch(p->at<void>(p->ly.wpk[l * 4 + 1]), p->tmA[1], dv.gs[1], y[1], err, o);
  if (e != cudaSuccess) return e;
  FM_REC(y[1], ybytes[1]);

  fm::RowArgs r1 = {};
  r1.M = c.M;
  r1.N = c.d;
  r1.parts = y[1];
  r1.nparts = dv.nparts(1);
  r1.sa = p->ascale(l, FM_SITE_ATTN_OUT);
  r1.sw = p->wscale(l, 1);
  r1.gate = p->mod(k, l, 2);
  r1.x = p->at<float>(p->ly.x);
  r1.do_quant = 1;
  r1.scale = p->mod(k, l, 3);
  r1.shift = p->mod(k, l, 4);
  r1.sq = p->ascale(l, FM_SITE_MLP_IN);
  r1.q = p->at<void>(p->ly.q2);
  r1.q_fp8 = fp8;
  r1.eps = c.rms_eps;
  if (!dv.rowfuse && !dv.ofuse) {
    e = fm::row_launch(r1, o);
    if (e != cudaSuccess) return e;
  }
  FM_REC(p->at<void>(p->ly.x), xbytes);
  if (!dv.rowfuse) FM_REC(p->at<void>(p->ly.q2), static_cast<size_t>(c.M) * c.d * ab);
  fm::GemmFuse fg = fq;   // the gate|up GEMM normalises and quantises with the pre-MLP norm
  fg.scale = p->mod(k, l, 3);
  fg.shift = p->mod(k, l, 4);
  fg.sqa = p->ascale(l, FM_SITE_MLP_IN);
  fg.q_out = p->at<void>(p->ly.q2);

  // gate|up: the epilogue applies GeGLU and quantises, writing the down GEMM's operand
  if (dv.nvfp4)
    e = fm::nvfp4_gemm_launch(p->tmA[2], p->at<void>(p->ly.wpk[l * 4 + 2]), dv.ns[2], nullptr, p->at<__half>(p->ly.mc),
                              p->ascale(l, FM_SITE_MLP_IN), p->wscale(l, 2), p->ascale(l, FM_SITE_GEGLU), err, o,
                              dv.act4);
  else
    // the gate|up GEMM's CTAs (two per SM) leave no room for most of the down GEMM's,
    // which then start late: with BF16 weights they find theirs in L2, prefetched here
    // after each CTA's own weight copies (FP8 down weights are half the bytes and come
    // in time without it; there the prefetch only adds traffic)
    e = fm::gemm_launch(p->at<void>(p->ly.wpk[l * 4 + 2]), p->tmA[2], dv.gs[2], nullptr, err, o, nullptr,
                        p->ascale(l, FM_SITE_MLP_IN), p->wscale(l, 2), p->at<void>(p->ly.mc), fp8,
                        p->ascale(l, FM_SITE_GEGLU), nullptr, nullptr, 0, 0, dv.rowfuse ? &fg : nullptr,
                        c.weight_fmt == FM_FMT_BF16 ? p->at<void>(p->ly.wpk[l * 4 + 3]) : nullptr,
                        c.weight_fmt == FM_FMT_BF16 ? fm::packed_weight_bytes(dv.gN[3], dv.gK[3], c.weight_fmt) : 0);
  if (e != cudaSuccess) return e;
  if (dv.rowfuse) FM_REC(p->at<void>(p->ly.q2), static_cast<size_t>(c.M) * c.d * ab);
  FM_REC(p->at<void>(p->ly.mc), static_cast<size_t>(c.M) * c.F * ab);

  fm::GemmFuse fd = fo;   // the down GEMM applies the MLP's gated residual itself
  fd.gate = p->mod(k, l, 5);
  if (dv.nvfp4)
    e = fm::nvfp4_gemm_launch(p->tmA[3], p->at<void>(p->ly.wpk[l * 4 + 3]), dv.ns[3], y[3], nullptr, nullptr, nullptr,
                              nullptr, err, o);
  else if (dv.rowfuse)
    e = fm::gemm_launch(p->at<void>(p->ly.wpk[l * 4 + 3]), p->tmA[3], dv.gs[3], nullptr, err, o, nullptr,
                        p->ascale(l, FM_SITE_GEGLU), p->wscale(l, 3), nullptr, 0, nullptr, nullptr, nullptr, 0, 0,
                        &fd);
  else
    e = fm::gemm_launch(p->at<void>(p->ly.wpk[l * 4 + 3]), p->tmA[3], dv.gs[3], y[3], err, o);
  if (e != cudaSuccess) return e;
  FM_REC(y[3], ybytes[3]);

  fm::RowArgs r2 = {};
  r2.M = c.M;
  r2.N = c.d;
  r2.parts = y[3];
  r2.nparts = dv.nparts(3);
  r2.sa = p->ascale(l, FM_SITE_GEGLU);
  r2.sw = p->wscale(l, 3);
  r2.gate = p->mod(k, l, 5);
  r2.x = p->at<float>(p->ly.x);
  r2.eps = c.rms_eps;
  r2.q = p->at<void>(p->ly.q);
  r2.q_fp8 = fp8;
  if (!step_end) {
    const int ln = (l + 1) % c.L;
    r2.do_quant = 1;
    r2.scale = p->mod(k, ln, 0);
    r2.shift = p->mod(k, ln, 1);
    r2.sq = p->ascale(ln, FM_SITE_ATTN_IN);
  } else {
    r2.do_tail = 1;
    r2.scale_f = p->modf(k, 0);
    r2.shift_f = p->modf(k, 1);
    r2.gamma_f = p->at<float>(p->ly.gamma_f);
    r2.w_out = p->at<__nv_bfloat16>(p->ly.w_out);
    r2.b_out = p->at<float>(p->ly.b_out);
    r2.a = p->at<float>(p->ly.a);
    r2.A = c.A;
    // step k < S of the schedule, or the warm start's single step (k == S) from warm_t
    r2.dt = k < c.S ? -1.0f / static_cast<float>(c.S) : -c.warm_t;
    if (k + 1 >= c.S) {   // the decision's last kernel
      r2.stamp = p->at<unsigned long long>(p->ly.stamps);
      r2.stamp_kind = 2;
    }
    if (k + 1 < c.S) {
      r2.do_head = 1;
      r2.w_in = p->at<__nv_bfloat16>(p->ly.w_in);
      r2.b_in = p->at<float>(p->ly.b_in);
      r2.do_quant = 1;
      r2.scale = p->mod(k + 1, 0, 0);
      r2.shift = p->mod(k + 1, 0, 1);
      r2.sq = p->ascale(0, FM_SITE_ATTN_IN);
    }
  }
  if (dv.rowfuse) {
    // the down GEMM already applied the residual; a step boundary still needs the
    // Euler tail (and the next step's head, whose x the next QKV GEMM normalises)
    r2.parts = nullptr;
    r2.do_quant = 0;
    r2.ssq = ssq;
    r2.ssq_tiles = c.d / 128;
  }
  if (!dv.rowfuse || step_end) {
    e = fm::row_launch(r2, o);
    if (e != cudaSuccess) return e;
  }
  FM_REC(p->at<void>(p->ly.x), xbytes);
  FM_REC(p->at<void>(p->ly.a), p->ly.a_bytes);
#undef FM_REC
  return cudaSuccess;
}

size_t trace_record_bytes(const fm_policy* p) {
  const fm_config& c = p->cfg;
  const Derived& dv = p->dv;
  const size_t M = c.M, ab = dv.act_bytes;
  size_t n = 3 * M * c.d * 4 + M * c.d * ab * 2 + M * c.H * c.Dh * ab + M * c.F * ab + p->ly.a_bytes;
  n += M * dv.gN[0] * (dv.attn_fp8 ? 1 : 2);
  for (int g = 1; g < 4; g += 2) n += static_cast<size_t>(dv.nparts(g)) * M * dv.gN[g] * 4;
  return n;
}

cudaError_t enqueue_head(fm_policy* p, const LaunchOpts& o, int k0 = 0) {
  const fm_config& c = p->cfg;
  fm::RowArgs r = {};
  r.M = c.M;
  r.N = c.d;
  r.x = p->at<float>(p->ly.x);
  r.a = p->at<float>(p->ly.a);
  r.A = c.A;
  r.do_head = 1;
  r.w_in = p->at<__nv_bfloat16>(p->ly.w_in);
  r.b_in = p->at<float>(p->ly.b_in);
  r.do_quant = 1;
  r.scale = p->mod(k0, 0, 0);
  r.shift = p->mod(k0, 0, 1);
  r.sq = p->ascale(0, FM_SITE_ATTN_IN);
  r.q = p->at<void>(p->ly.q);
  r.q_fp8 = p->dv.q_store;
  r.eps = c.rms_eps;
  r.stamp = p->at<unsigned long long>(p->ly.stamps);
  r.stamp_kind = 1;
  if (p->dv.rowfuse) {   // the first QKV GEMM normalises x itself: hand it the row sums
    r.do_quant = 0;
    r.ssq = p->at<float>(p->ly.ssq);
    r.ssq_tiles = c.d / 128;
  }
  return fm::row_launch(r, o);
}

cudaError_t enqueue_decision(fm_policy* p, cudaStream_t st, Trace* tr = nullptr, unsigned long long* tl = nullptr) {
  LaunchOpts o;
  o.stream = st;
  o.pdl = (p->cfg.flags & FM_FLAG_USE_PDL) != 0;
  o.tl = tl;
  cudaError_t e = enqueue_head(p, o);
  if (e != cudaSuccess) return e;
  for (int k = 0; k < p->cfg.S; ++k)
    for (int l = 0; l < p->cfg.L; ++l) {
      e = enqueue_layer(p, l, k, l == p->cfg.L - 1, o, tr);
      if (e != cudaSuccess) return e;
    }
  return cudaGetLastError();
}

// The warm start's single step: the head and all layers with modulation row S; the
// last layer's tail steps by dt = -warm_t.
cudaError_t enqueue_warm_traced(fm_policy* p, cudaStream_t st, Trace* tr) {
  LaunchOpts o;
  o.stream = st;
  o.pdl = (p->cfg.flags & FM_FLAG_USE_PDL) != 0;
  cudaError_t e = enqueue_head(p, o, p->cfg.S);
  if (e != cudaSuccess) return e;
  for (int l = 0; l < p->cfg.L; ++l) {
    e = enqueue_layer(p, l, p->cfg.S, l == p->cfg.L - 1, o, tr);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t enqueue_warm(fm_policy* p, cudaStream_t st) { return enqueue_warm_traced(p, st, nullptr); }

int capture(fm_policy* p, cudaError_t (*enq)(fm_policy*, cudaStream_t), cudaGraph_t* graph, cudaGraphExec_t* exec,
            const char* what) {
  FM_CUDA(p, cudaStreamBeginCapture(p->cap_stream, cudaStreamCaptureModeThreadLocal));
  cudaError_t e = enq(p, p->cap_stream);
  cudaGraph_t g = nullptr;
  cudaError_t e2 = cudaStreamEndCapture(p->cap_stream, &g);
  if (e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return cuda_fail(p, e, what);
  }
  if (e2 != cudaSuccess) return cuda_fail(p, e2, "cudaStreamEndCapture");
  *graph = g;
  FM_CUDA(p, cudaGraphInstantiate(exec, g, 0));
  return FM_OK;
}

cudaError_t enqueue_full(fm_policy* p, cudaStream_t st) { return enqueue_decision(p, st); }

int build_graph(fm_policy* p) {
  FM_CUDA(p, cudaStreamCreateWithFlags(&p->cap_stream, cudaStreamNonBlocking));
  int st = capture(p, enqueue_full, &p->graph, &p->exec, "capturing the decision");
  if (st != FM_OK || !(p->cfg.warm_t > 0.f)) return st;
  return capture(p, enqueue_warm, &p->warm_graph, &p->warm_exec, "capturing the warm start");
}

void release(fm_policy* p) {
  if (!p) return;
  if (p->exec) cudaGraphExecDestroy(p->exec);
  if (p->graph) cudaGraphDestroy(p->graph);
  if (p->warm_exec) cudaGraphExecDestroy(p->warm_exec);
  if (p->warm_graph) cudaGraphDestroy(p->warm_graph);
  if (p->cap_stream) cudaStreamDestroy(p->cap_stream);
  delete p;
}

// Tensor maps of the GEMM activation operands (fixed addresses, recorded into the
// graph by value); packed weights are fetched with plain bulk copies.
bool build_tmaps(fm_policy* p) {
  const size_t act_off[4] = {p->ly.q, p->ly.o, p->ly.q2, p->ly.mc};
  for (int g = 0; g < 4; ++g) {
    const bool ok = p->dv.nvfp4 ? fm::nvfp4_tmap_act(&p->tmA[g], p->at<void>(act_off[g]), p->dv.ns[g])
                                : fm::gemm_tmap_act(&p->tmA[g], p->at<void>(act_off[g]), p->dv.gs[g]);
    if (!ok) return false;
  }
  if (p->dv.ofuse && !fm::o_consumer_tmap(&p->tmO, p->at<void>(p->ly.o), p->dv.os)) return false;
  return true;
}

int check_ptrs(const fm_weights* w, int L, bool given, std::string* why) {
  if (!w || !w->layers || !w->w_in || !w->b_in || !w->w_out || !w->b_out || !w->gamma_f || !w->w_mod_f ||
      !w->b_mod_f || (given && !w->conds)) {
    *why = "a weight pointer is NULL";
    return FM_ERR_INVALID_ARG;
  }
  for (int l = 0; l < L; ++l) {
    const fm_layer_weights& lw = w->layers[l];
    const void* ptrs[8] = {lw.w_qkv, lw.w_o, lw.w_gu, lw.w_d, lw.gamma1, lw.gamma2, lw.w_mod, lw.b_mod};
    for (const void* q : ptrs) {
      if (!q) {
        *why = "a layer weight pointer is NULL";
        return FM_ERR_INVALID_ARG;
      }
      if (!aligned16(q)) {
        *why = "a layer weight pointer is not 16-byte aligned";
        return FM_ERR_ALIGN;
      }
    }
  }
  const void* ptrs[7] = {w->w_in, w->b_in, w->w_out, w->b_out, w->gamma_f, w->w_mod_f, w->b_mod_f};
  for (const void* q : ptrs)
    if (!aligned16(q)) {
      *why = "a weight pointer is not 16-byte aligned";
      return FM_ERR_ALIGN;
    }
  return FM_OK;
}

}  // namespace

namespace fm {

int record_error(int status, const char* why) { return fail(nullptr, status, why); }

int gemm_consumer_scratch_bytes(int M, int N, int K, int fmt, int s, size_t* bytes, const char** why) {
  if (fmt != FM_FMT_FP8 && fmt != FM_FMT_BF16) {
    *why = "fmt must be FM_FMT_FP8 or FM_FMT_BF16";
    return FM_ERR_INVALID_ARG;
  }
  GemmShape g;
  if (gemm_plan(M, N, K, fmt == FM_FMT_FP8, s, cluster_for(s), &g) != FM_OK || N > 16384) {
    *why = "shape: 1 <= M <= 256, N and K multiples of 128, N <= 16384, s dividing the K-block count";
    return FM_ERR_SHAPE;
  }
  *bytes = static_cast<size_t>(g.s / g.cs) * M * N * sizeof(float);
  return FM_OK;
}

int gemm_consumer_run(const GemmConsumerArgs& a, float* scratch, size_t scratch_bytes, int* err_word,
                      cudaStream_t st, const char** why) {
  if (!a.a || !a.w_packed || !a.s_a || !a.s_w || !a.x || !a.gate || !a.scale || !a.shift || !a.s_q || !a.q ||
      !scratch) {
    *why = "NULL argument";
    return FM_ERR_INVALID_ARG;
  }
  size_t need = 0;
  const int st0 = gemm_consumer_scratch_bytes(a.M, a.N, a.K, a.fmt, a.s, &need, why);
  if (st0 != FM_OK) return st0;
  if (scratch_bytes < need) {
    *why = "scratch smaller than the split-K partial planes need";
    return FM_ERR_WORKSPACE;
  }
  const void* ptrs[8] = {a.a, a.x, a.gate, a.scale, a.shift, a.q, scratch, a.bias ? a.bias : a.x};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) {
      *why = "pointers must be 16-byte aligned";
      return FM_ERR_ALIGN;
    }
  if (reinterpret_cast<uintptr_t>(a.w_packed) % kAlign) {
    *why = "w_packed must be 1024-byte aligned";
    return FM_ERR_ALIGN;
  }
  GemmShape g;
  gemm_plan(a.M, a.N, a.K, a.fmt == FM_FMT_FP8, a.s, cluster_for(a.s), &g);
  CUtensorMap ta;
  if (!gemm_tmap_act(&ta, a.a, g)) {
    *why = "cuTensorMapEncodeTiled failed";
    return FM_ERR_CUDA;
  }
  if (gemm_configure() != cudaSuccess) {
    *why = "configuring the GEMM kernels failed";
    return FM_ERR_CUDA;
  }
  LaunchOpts o;
  o.stream = st;
  if (gemm_launch(a.w_packed, ta, g, scratch, err_word, o) != cudaSuccess) {
    *why = "GEMM launch failed";
    return FM_ERR_CUDA;
  }
  RowArgs r = {};
  r.M = a.M;
  r.N = a.N;
  r.parts = scratch;
  r.nparts = g.s / g.cs;
  r.sa = a.s_a;
  r.sw = a.s_w;
  r.bias = a.bias;
  r.gate = a.gate;
  r.x = a.x;
  r.do_quant = 1;
  r.scale = a.scale;
  r.shift = a.shift;
  r.sq = a.s_q;
  r.q = a.q;
  r.q_fp8 = a.fmt == FM_FMT_FP8;
  r.eps = a.eps;
  if (row_launch(r, o) != cudaSuccess) {
    *why = "consumer launch failed";
    return FM_ERR_CUDA;
  }
  return FM_OK;
}

}  // namespace fm

// ==================================================================== C ABI
extern "C" {

const char* fm_status_string(int s) {
  switch (s) {
    case FM_OK: return "FM_OK";
    case FM_ERR_INVALID_ARG: return "FM_ERR_INVALID_ARG";
    case FM_ERR_SHAPE: return "FM_ERR_SHAPE";
    case FM_ERR_ALIGN: return "FM_ERR_ALIGN";
    case FM_ERR_WORKSPACE: return "FM_ERR_WORKSPACE";
    case FM_ERR_CUDA: return "FM_ERR_CUDA";
    case FM_ERR_STATE_MISMATCH: return "FM_ERR_STATE_MISMATCH";
    case FM_ERR_DEVICE: return "FM_ERR_DEVICE";
    case FM_ERR_UNSUPPORTED: return "FM_ERR_UNSUPPORTED";
    default: return "FM_ERR_UNKNOWN";
  }
}

const char* fm_last_error(const fm_policy* p) { return p ? p->err.c_str() : g_last_error.c_str(); }

int fm_abi_sizes(size_t* config, size_t* weights, size_t* layer_weights, size_t* timing) {
  if (config) *config = sizeof(fm_config);
  if (weights) *weights = sizeof(fm_weights);
  if (layer_weights) *layer_weights = sizeof(fm_layer_weights);
  if (timing) *timing = sizeof(fm_timing);
  return FM_OK;
}

int fm_workspace_size(const fm_config* cfg, size_t* bytes) {
  std::string why;
  int st = validate(cfg, &why);
  if (st != FM_OK) return fail(nullptr, st, why);
  if (!bytes) return fail(nullptr, FM_ERR_INVALID_ARG, "bytes is NULL");
  Derived dv;
  st = derive(cfg, &dv, &why);
  if (st != FM_OK) return fail(nullptr, st, why);
  *bytes = make_layout(cfg, dv).total;
  return FM_OK;
}

int policy_create(const fm_config* cfg, const fm_weights* w, const float* act_scales, void* workspace,
                  size_t ws_bytes, void* stream, fm_policy** out) {
  if (!out) return fail(nullptr, FM_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  std::string why;
  int st = validate(cfg, &why);
  if (st != FM_OK) return fail(nullptr, st, why);
  st = check_ptrs(w, cfg->L, cfg->cond_mode == FM_COND_GIVEN, &why);
  if (st != FM_OK) return fail(nullptr, st, why);
  if ((cfg->act_fmt == FM_FMT_FP8 || cfg->act_fmt == FM_FMT_NVFP4) && !act_scales)
    return fail(nullptr, FM_ERR_INVALID_ARG, "FP8 and four-bit activations need an activation-scale table");
  if (!workspace) return fail(nullptr, FM_ERR_INVALID_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return fail(nullptr, FM_ERR_ALIGN, "workspace not 1024-aligned");

  fm_policy* p = new (std::nothrow) fm_policy();
  if (!p) return fail(nullptr, FM_ERR_INVALID_ARG, "out of host memory");
  p->cfg = *cfg;
  st = derive(cfg, &p->dv, &why);
  if (st != FM_OK) {
    release(p);
    return fail(nullptr, st, why);
  }
  p->ly = make_layout(cfg, p->dv);
  if (ws_bytes < p->ly.total) {
    char buf[128];
    snprintf(buf, sizeof buf, "workspace has %zu bytes, needs %zu", ws_bytes, p->ly.total);
    release(p);
    return fail(nullptr, FM_ERR_WORKSPACE, buf);
  }
  p->ws = static_cast<uint8_t*>(workspace);
  p->ws_bytes = ws_bytes;
  p->shared = p->ws;
  p->state = p->ws + p->ly.shared_end;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const fm_config& c = p->cfg;
  const Derived& dv = p->dv;

  auto bail = [&](int code, const std::string& msg) {
    release(p);
    return fail(nullptr, code, msg);
  };
  auto cu = [&](cudaError_t e, const char* where) -> bool {
    if (e == cudaSuccess) return true;
    why = std::string(where) + ": " + cudaGetErrorString(e);
    return false;
  };

  if (!cu(fm::gemm_configure(), "gemm_configure") || !cu(fm::nvfp4_configure(), "nvfp4_configure") ||
      !cu(fm::attn_configure(), "attn_configure") || !cu(fm::o_consumer_configure(), "o_consumer_configure"))
    return bail(FM_ERR_CUDA, why);

  // weights: fold gamma, quantise, tile
  unsigned* amax = p->at<unsigned>(p->ly.amax);
  for (int l = 0; l < c.L; ++l) {
    const fm_layer_weights& lw = w->layers[l];
    const float* src[4] = {lw.w_qkv, lw.w_o, lw.w_gu, lw.w_d};
    const float* gam[4] = {lw.gamma1, nullptr, lw.gamma2, nullptr};
    for (int g = 0; g < 4; ++g) {
      if (!cu(fm::pack_weight(src[g], gam[g], dv.gN[g], dv.gK[g], c.weight_fmt, p->at<void>(p->ly.wpk[l * 4 + g]),
                              p->wscale(l, g), amax, s, g == 2),
              "pack_weight"))
        return bail(FM_ERR_CUDA, why);
    }
  }
  // modulation table (the t-schedule is fixed: per-create state)
  double* conds = p->at<double>(p->ly.conds);
  const int mod_rows = c.S + (c.warm_t > 0.f ? 1 : 0);
  if (!cu(fm::cond_embed_launch(conds, c.S, c.d, c.cond_mode == FM_COND_GIVEN ? w->conds : nullptr, c.warm_t, s),
          "cond_embed"))
    return bail(FM_ERR_CUDA, why);
  for (int l = 0; l < c.L; ++l) {
    const fm_layer_weights& lw = w->layers[l];
    if (!cu(fm::modtable_launch(conds, mod_rows, c.d, reinterpret_cast<const __nv_bfloat16*>(lw.w_mod), lw.b_mod, 6 * c.d,
                                p->mod(0, l, 0), static_cast<size_t>(c.L) * 6 * c.d, s),
            "modtable"))
      return bail(FM_ERR_CUDA, why);
  }
  if (!cu(fm::modtable_launch(conds, mod_rows, c.d, reinterpret_cast<const __nv_bfloat16*>(w->w_mod_f), w->b_mod_f,
                              2 * c.d, p->modf(0, 0), static_cast<size_t>(2) * c.d, s),
          "modtable_final"))
    return bail(FM_ERR_CUDA, why);
  // in/out projections
  const size_t da = static_cast<size_t>(c.d) * c.A;
  if (!cu(cudaMemcpyAsync(p->at<void>(p->ly.w_in), w->w_in, da * 2, cudaMemcpyDeviceToDevice, s), "copy w_in") ||
      !cu(cudaMemcpyAsync(p->at<void>(p->ly.w_out), w->w_out, da * 2, cudaMemcpyDeviceToDevice, s), "copy w_out") ||
      !cu(cudaMemcpyAsync(p->at<void>(p->ly.b_in), w->b_in, c.d * 4, cudaMemcpyDeviceToDevice, s), "copy b_in") ||
      !cu(cudaMemcpyAsync(p->at<void>(p->ly.b_out), w->b_out, c.A * 4, cudaMemcpyDeviceToDevice, s), "copy b_out") ||
      !cu(cudaMemcpyAsync(p->at<void>(p->ly.gamma_f), w->gamma_f, c.d * 4, cudaMemcpyDeviceToDevice, s),
          "copy gamma_f"))
    return bail(FM_ERR_CUDA, why);
  // activation scales (BF16 activations: 1)
  const std::vector<float> sc = scale_table(c, dv, act_scales);
  if (!cu(cudaMemcpyAsync(p->at<void>(p->ly.ascale), sc.data(), sc.size() * 4, cudaMemcpyHostToDevice, s),
          "copy act scales") ||
      !cu(cudaMemsetAsync(p->at<void>(p->ly.kcache), 0, p->ly.kv_bytes, s), "zero kcache") ||
      !cu(cudaMemsetAsync(p->at<void>(p->ly.vcache), 0, p->ly.kv_bytes, s), "zero vcache") ||
      !cu(cudaMemsetAsync(p->at<void>(p->ly.kcache8), 0, std::max<size_t>(p->ly.kv8_bytes, 1), s), "zero kcache8") ||
      !cu(cudaMemsetAsync(p->at<void>(p->ly.vcache8), 0, std::max<size_t>(p->ly.v8_bytes, 1), s), "zero vcache8") ||
      !cu(cudaMemsetAsync(p->at<void>(p->ly.a), 0, p->ly.a_bytes, s), "zero a") ||
      !cu(cudaMemsetAsync(p->errw(), 0, 64, s), "zero err"))
    return bail(FM_ERR_CUDA, why);
  if (!cu(cudaStreamSynchronize(s), "create sync")) return bail(FM_ERR_CUDA, why);

  if (!build_tmaps(p)) return bail(FM_ERR_CUDA, "cuTensorMapEncodeTiled (activations) failed");

  uint64_t h = 1469598103934665603ull;
  h = fnv(h, &c, sizeof c);
  const uintptr_t base = reinterpret_cast<uintptr_t>(p->ws);
  h = fnv(h, &base, sizeof base);
  for (int g = 0; g < 4; ++g) h = fnv(h, &dv.gs[g], sizeof(fm::GemmShape));
  for (int g = 0; g < 4; ++g) h = fnv(h, &dv.ns[g], sizeof(fm::Nvfp4Shape));
  h = fnv(h, &dv.rowfuse, sizeof(int));
  h = fnv(h, &dv.attn_kc, sizeof(int));
  p->plan_hash = h;

  if (c.flags & FM_FLAG_USE_GRAPH) {
    st = build_graph(p);
    if (st != FM_OK) {
      why = p->err;
      return bail(st, why);
    }
  }
  *out = p;
  return FM_OK;
}

int policy_destroy(fm_policy* p) {
  if (!p) return fail(nullptr, FM_ERR_INVALID_ARG, "policy is NULL");
  if (p->sessions > 0) return fail(p, FM_ERR_INVALID_ARG, "the policy still has live sessions");
  if (p->base) --p->base->sessions;
  release(p);
  return FM_OK;
}

int fm_session_workspace_size(const fm_policy* base, size_t* bytes) {
  if (!base || !bytes) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL argument");
  *bytes = base->ly.total - base->ly.shared_end;
  return FM_OK;
}

int fm_session_create(fm_policy* base, void* workspace, size_t ws_bytes, void* stream, fm_policy** out) {
  if (!out) return fail(nullptr, FM_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!base || !workspace) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL argument");
  if (base->base) base = base->base;   // a session of a session shares the same weights
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return fail(nullptr, FM_ERR_ALIGN, "workspace not 1024-aligned");
  const size_t need = base->ly.total - base->ly.shared_end;
  if (ws_bytes < need) {
    char buf[128];
    snprintf(buf, sizeof buf, "session workspace has %zu bytes, needs %zu", ws_bytes, need);
    return fail(nullptr, FM_ERR_WORKSPACE, buf);
  }
  fm_policy* p = new (std::nothrow) fm_policy();
  if (!p) return fail(nullptr, FM_ERR_INVALID_ARG, "out of host memory");
  p->cfg = base->cfg;
  p->dv = base->dv;
  p->ly = base->ly;
  p->ws = static_cast<uint8_t*>(workspace);
  p->ws_bytes = ws_bytes;
  p->shared = base->shared;
  p->state = p->ws;
  p->plan_hash = base->plan_hash;   // the same plan: capsules move between its sessions by fork
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // fresh state: empty prefix cache, zero action buffer and error word; the base's
  // current activation scales
  cudaError_t e = cudaMemsetAsync(p->state, 0, need, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(p->at<void>(p->ly.ascale), base->at<void>(base->ly.ascale), p->ly.ascale_bytes,
                        cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    release(p);
    return fail(nullptr, FM_ERR_CUDA, std::string("session state init: ") + cudaGetErrorString(e));
  }
  if (!build_tmaps(p)) {
    release(p);
    return fail(nullptr, FM_ERR_CUDA, "cuTensorMapEncodeTiled (activations) failed");
  }
  if (p->cfg.flags & FM_FLAG_USE_GRAPH) {
    const int st = build_graph(p);
    if (st != FM_OK) {
      const std::string why = p->err;
      release(p);
      return fail(nullptr, st, why);
    }
  }
  p->base = base;
  ++base->sessions;
  *out = p;
  return FM_OK;
}

int fm_set_act_scales(fm_policy* p, const float* act_scales, void* stream) {
  if (!p || !act_scales) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  if (!p->dv.fp8 && !p->dv.act4) return FM_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const std::vector<float> sc = scale_table(p->cfg, p->dv, act_scales);
  FM_CUDA(p, cudaMemcpyAsync(p->at<void>(p->ly.ascale), sc.data(), sc.size() * 4, cudaMemcpyHostToDevice, s));
  if (p->dv.attn_fp8 && p->cfg.P > 0) FM_CUDA(p, requant_prefix(p, 0, p->cfg.P, s));
  return cudaStreamSynchronize(s) == cudaSuccess ? FM_OK : fail(p, FM_ERR_CUDA, "sync");
}

int set_prefix_kv(fm_policy* p, const uint16_t* k, const uint16_t* v, void* stream) {
  if (!p || !k || !v) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  if (p->cfg.P == 0) return FM_OK;
  return refresh_prefix(p, 0, p->cfg.P, k, v, stream);
}

int refresh_prefix(fm_policy* p, int tok_begin, int tok_end, const uint16_t* k, const uint16_t* v, void* stream) {
  if (!p || !k || !v) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  const fm_config& c = p->cfg;
  if (tok_begin < 0 || tok_end > c.P || tok_begin >= tok_end) return fail(p, FM_ERR_SHAPE, "bad token range");
  const size_t row = static_cast<size_t>(c.Hkv) * c.Dh * 2;
  const size_t rows = static_cast<size_t>(tok_end - tok_begin);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* kdst = p->at<uint8_t>(p->ly.kcache) + tok_begin * row;
  FM_CUDA(p, cudaMemcpy2DAsync(kdst, static_cast<size_t>(c.P) * row, k, rows * row, rows * row, c.L,
                               cudaMemcpyDeviceToDevice, s));
  // values are kept transposed, [L][Hkv][Dh][P_pad], the layout attention's P.V operand needs
  FM_CUDA(p, fm::transpose_v_launch(reinterpret_cast<const __nv_bfloat16*>(v), p->at<__nv_bfloat16>(p->ly.vcache), c.L,
                                    static_cast<int>(rows), c.Hkv, (c.P + 7) / 8 * 8, tok_begin, s));
  if (p->dv.attn_fp8) FM_CUDA(p, requant_prefix(p, tok_begin, tok_end, s));
  return FM_OK;
}

uint64_t steady_ns() {
  return static_cast<uint64_t>(std::chrono::duration_cast<std::chrono::nanoseconds>(
                                   std::chrono::steady_clock::now().time_since_epoch())
                                   .count());
}

int decode_actions(fm_policy* p, const float* noise, float* actions, void* stream) {
  if (!p || !actions) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* a = p->at<float>(p->ly.a);
  p->host_submit_ns = steady_ns();
  if (noise && noise != a) FM_CUDA(p, cudaMemcpyAsync(a, noise, p->ly.a_bytes, cudaMemcpyDeviceToDevice, s));
  if (p->exec) {
    FM_CUDA(p, cudaGraphLaunch(p->exec, s));
  } else {
    FM_CUDA(p, enqueue_decision(p, s));
  }
  if (actions != a) FM_CUDA(p, cudaMemcpyAsync(actions, a, p->ly.a_bytes, cudaMemcpyDeviceToDevice, s));
  ++p->decisions;
  p->have_prev = true;
  return FM_OK;
}

int fm_decode_warm(fm_policy* p, const float* noise, int executed, float* actions, void* stream) {
  if (!p || !noise || !actions) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  const fm_config& c = p->cfg;
  if (!(c.warm_t > 0.f)) return fail(p, FM_ERR_UNSUPPORTED, "the policy was created with warm_t = 0");
  if (executed < 0 || executed > c.M) return fail(p, FM_ERR_INVALID_ARG, "executed must lie in [0, M]");
  if (!p->have_prev) return decode_actions(p, noise, actions, stream);   // episode start: all S steps
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* a = p->at<float>(p->ly.a);
  float* prev = p->at<float>(p->ly.prev);
  p->host_submit_ns = steady_ns();
  FM_CUDA(p, cudaMemcpyAsync(prev, a, p->ly.a_bytes, cudaMemcpyDeviceToDevice, s));
  FM_CUDA(p, fm::warm_mix_launch(a, prev, noise, c.M, c.A, executed, c.warm_t, s));
  if (p->warm_exec) {
    FM_CUDA(p, cudaGraphLaunch(p->warm_exec, s));
  } else {
    FM_CUDA(p, enqueue_warm(p, s));
  }
  if (actions != a) FM_CUDA(p, cudaMemcpyAsync(actions, a, p->ly.a_bytes, cudaMemcpyDeviceToDevice, s));
  ++p->decisions;
  return FM_OK;
}

int fm_episode_reset(fm_policy* p) {
  if (!p) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL policy");
  p->have_prev = false;
  return FM_OK;
}

int fm_decode_actions_seeded(fm_policy* p, uint64_t seed, uint64_t counter, float* actions, void* stream) {
  if (!p || !actions) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* a = p->at<float>(p->ly.a);
  FM_CUDA(p, fm::philox_noise_launch(a, static_cast<int64_t>(p->cfg.M) * p->cfg.A, seed, counter, nullptr, s));
  return decode_actions(p, nullptr, actions, stream);
}

int fm_philox_noise(float* out, int64_t n, uint64_t seed, uint64_t counter, uint32_t* raw_words, void* stream) {
  if (!out || n < 0) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL output or negative size");
  const cudaError_t e = fm::philox_noise_launch(out, n, seed, counter, raw_words, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(nullptr, FM_ERR_CUDA, cudaGetErrorString(e));
  return FM_OK;
}

int fm_last_timing(fm_policy* p, fm_timing* t, void* stream) {
  if (!p || !t) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long st[2] = {0, 0};
  FM_CUDA(p, cudaMemcpyAsync(st, p->at<void>(p->ly.stamps), sizeof st, cudaMemcpyDeviceToHost, s));
  FM_CUDA(p, cudaStreamSynchronize(s));
  t->host_submit_ns = p->host_submit_ns;
  t->device_start_ns = st[0];
  t->device_end_ns = st[1];
  return FM_OK;
}

int decode_actions_host(fm_policy* p, const float* noise_host, float* actions_host, void* stream) {
  if (!p || !actions_host) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* a = p->at<float>(p->ly.a);
  if (noise_host) FM_CUDA(p, cudaMemcpyAsync(a, noise_host, p->ly.a_bytes, cudaMemcpyHostToDevice, s));
  const int st = decode_actions(p, nullptr, a, stream);
  if (st != FM_OK) return st;
  FM_CUDA(p, cudaMemcpyAsync(actions_host, a, p->ly.a_bytes, cudaMemcpyDeviceToHost, s));
  FM_CUDA(p, cudaStreamSynchronize(s));
  return FM_OK;
}

int fm_state_size(const fm_policy* p, size_t* bytes) {
  if (!p || !bytes) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL argument");
  *bytes = sizeof(CapsuleHeader) + 2 * p->ly.kv_bytes + p->ly.a_bytes + p->ly.ascale_bytes;
  return FM_OK;
}

int snapshot_state(fm_policy* p, void* dst, size_t bytes, int dst_on_device, void* stream) {
  if (!p || !dst) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  size_t need = 0;
  fm_state_size(p, &need);
  if (bytes < need) return fail(p, FM_ERR_WORKSPACE, "capsule buffer too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CapsuleHeader& h = p->hdr;
  std::memset(&h, 0, sizeof h);
  h.magic = kCapsuleMagic;
  h.abi = FM_ABI_VERSION;
  h.header_bytes = sizeof h;
  h.plan_hash = p->plan_hash;
  h.ws_base = reinterpret_cast<uintptr_t>(p->ws);
  h.kv_bytes = p->ly.kv_bytes;
  h.a_bytes = p->ly.a_bytes;
  h.scale_bytes = p->ly.ascale_bytes;
  h.L = p->cfg.L;
  h.P = p->cfg.P;
  h.Hkv = p->cfg.Hkv;
  h.Dh = p->cfg.Dh;
  h.M = p->cfg.M;
  h.A = p->cfg.A;
  h.decisions = p->decisions;
  uint8_t* d = static_cast<uint8_t*>(dst);
  const cudaMemcpyKind k = dst_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost;
  if (dst_on_device) {
    FM_CUDA(p, cudaMemcpyAsync(d, &h, sizeof h, cudaMemcpyHostToDevice, s));
    FM_CUDA(p, cudaStreamSynchronize(s));   // the staging header is reused by the next snapshot
  } else {
    std::memcpy(d, &h, sizeof h);
  }
  size_t off = sizeof h;
  const size_t regions[4][2] = {{p->ly.kcache, p->ly.kv_bytes},
                                {p->ly.vcache, p->ly.kv_bytes},
                                {p->ly.a, p->ly.a_bytes},
                                {p->ly.ascale, p->ly.ascale_bytes}};
  for (const auto& r : regions) {
    if (r[1]) FM_CUDA(p, cudaMemcpyAsync(d + off, p->at<void>(r[0]), r[1], k, s));
    off += r[1];
  }
  if (!dst_on_device) FM_CUDA(p, cudaStreamSynchronize(s));
  return FM_OK;
}

static int restore_impl(fm_policy* p, const void* src, size_t bytes, int src_on_device, void* stream, bool bound);

int restore_state(fm_policy* p, const void* src, size_t bytes, int src_on_device, void* stream) {
  return restore_impl(p, src, bytes, src_on_device, stream, true);
}

int fm_session_fork(fm_policy* base, const void* capsule, size_t bytes, int capsule_on_device, void* workspace,
                    size_t ws_bytes, void* stream, fm_policy** out) {
  if (!out) return fail(nullptr, FM_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!base || !capsule) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL argument");
  fm_policy* p = nullptr;
  int st = fm_session_create(base, workspace, ws_bytes, stream, &p);
  if (st != FM_OK) return st;
  st = restore_impl(p, capsule, bytes, capsule_on_device, stream, false);
  if (st != FM_OK) {
    const std::string why = p->err;
    policy_destroy(p);
    return fail(nullptr, st, why);
  }
  *out = p;
  return FM_OK;
}

static int restore_impl(fm_policy* p, const void* src, size_t bytes, int src_on_device, void* stream, bool bound) {
  if (!p || !src) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  size_t need = 0;
  fm_state_size(p, &need);
  if (bytes < need) return fail(p, FM_ERR_STATE_MISMATCH, "capsule too small for this policy");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CapsuleHeader h;
  if (src_on_device) {
    FM_CUDA(p, cudaMemcpyAsync(&h, src, sizeof h, cudaMemcpyDeviceToHost, s));
    FM_CUDA(p, cudaStreamSynchronize(s));
  } else {
    std::memcpy(&h, src, sizeof h);
  }
  if (h.magic != kCapsuleMagic || h.abi != FM_ABI_VERSION || h.header_bytes != sizeof h)
    return fail(p, FM_ERR_STATE_MISMATCH, "not a capsule of this library version");
  if (h.plan_hash != p->plan_hash) return fail(p, FM_ERR_STATE_MISMATCH, "capsule was made by another plan");
  if (bound && h.ws_base != reinterpret_cast<uintptr_t>(p->ws))
    return fail(p, FM_ERR_STATE_MISMATCH, "capsule is bound to another workspace address");
  if (h.kv_bytes != p->ly.kv_bytes || h.a_bytes != p->ly.a_bytes || h.scale_bytes != p->ly.ascale_bytes ||
      h.L != p->cfg.L || h.P != p->cfg.P || h.M != p->cfg.M || h.A != p->cfg.A)
    return fail(p, FM_ERR_STATE_MISMATCH, "capsule shapes differ");
  const uint8_t* sp = static_cast<const uint8_t*>(src);
  const cudaMemcpyKind k = src_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
  size_t off = sizeof h;
  const size_t regions[4][2] = {{p->ly.kcache, p->ly.kv_bytes},
                                {p->ly.vcache, p->ly.kv_bytes},
                                {p->ly.a, p->ly.a_bytes},
                                {p->ly.ascale, p->ly.ascale_bytes}};
  for (const auto& r : regions) {
    if (r[1]) FM_CUDA(p, cudaMemcpyAsync(p->at<void>(r[0]), sp + off, r[1], k, s));
    off += r[1];
  }
  // the E4M3 prefix copy is derived state: re-derive it from the restored cache and scales
  if (p->dv.attn_fp8 && p->cfg.P > 0) FM_CUDA(p, requant_prefix(p, 0, p->cfg.P, s));
  if (!src_on_device) FM_CUDA(p, cudaStreamSynchronize(s));
  p->decisions = h.decisions;
  p->have_prev = h.decisions > 0;   // the restored noise/action buffer holds a decided chunk
  return FM_OK;
}

int fm_device_status(fm_policy* p, void* stream, int* word) {
  if (!p || !word) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int w = 0;
  FM_CUDA(p, cudaMemcpyAsync(&w, p->errw(), sizeof w, cudaMemcpyDeviceToHost, s));
  FM_CUDA(p, cudaMemsetAsync(p->errw(), 0, sizeof w, s));
  FM_CUDA(p, cudaStreamSynchronize(s));
  *word = w;
  return w ? fail(p, FM_ERR_DEVICE, "a kernel abandoned a bounded wait") : FM_OK;
}

int fm_standalone_status(void* stream, int* word) {
  if (!word) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  int* words[2] = {nullptr, nullptr};
  FM_CUDA(nullptr, cudaGetDevice(&dev));
  FM_CUDA(nullptr, cudaGetSymbolAddress(reinterpret_cast<void**>(&words[0]), fm_standalone_err));
  words[1] = fm::noalloc_error_word(dev);
  int got[2] = {0, 0};
  for (int i = 0; i < 2; ++i) {
    if (!words[i]) continue;
    FM_CUDA(nullptr, cudaMemcpyAsync(&got[i], words[i], sizeof(int), cudaMemcpyDeviceToHost, s));
    FM_CUDA(nullptr, cudaMemsetAsync(words[i], 0, sizeof(int), s));
  }
  FM_CUDA(nullptr, cudaStreamSynchronize(s));
  *word = got[0] | got[1];
  return *word ? fail(nullptr, FM_ERR_DEVICE, "a standalone kernel abandoned a bounded wait") : FM_OK;
}

int fm_named_buffer(const fm_policy* p, const char* name, void** ptr, size_t* bytes) {
  if (!p || !name || !ptr || !bytes) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL argument");
  const fm_config& c = p->cfg;
  const Derived& dv = p->dv;
  const Layout& ly = p->ly;
  const size_t M = c.M, ab = dv.act_bytes;
  auto ypart = [&](int g) { return static_cast<size_t>(dv.nparts(g)) * M * dv.gN[g] * 4; };
  struct Entry {
    const char* n;
    size_t off, bytes;
  } table[] = {
      {"prefix_k", ly.kcache, ly.kv_bytes},
      {"prefix_v", ly.vcache, ly.kv_bytes},
      {"actions", ly.a, ly.a_bytes},
      {"x", ly.x, M * c.d * 4},
      {"q", ly.q, M * c.d * ab},
      {"q2", ly.q2, M * c.d * ab},
      {"attn_out", ly.o, M * c.H * c.Dh * ab},
      {"geglu_out", ly.mc, M * c.F * ab},
      {"y_qkv", ly.qkvb, M * dv.gN[0] * 2},
      {"y_o", ly.y[1], ypart(1)},
      {"y_d", ly.y[3], ypart(3)},
      {"act_scales", ly.ascale, ly.ascale_bytes},
      {"prefix_k8", ly.kcache8, ly.kv8_bytes},
      {"prefix_v8", ly.vcache8, ly.v8_bytes},
      {"weight_scales", ly.wscale, ly.scale_bytes},
      {"mod", ly.mod, static_cast<size_t>(c.S) * c.L * 6 * c.d * 4},
      {"mod_final", ly.modf, static_cast<size_t>(c.S) * 2 * c.d * 4},
  };
  for (const Entry& e : table) {
    if (std::strcmp(e.n, name) == 0) {
      *ptr = p->at<uint8_t>(e.off);
      *bytes = e.bytes;
      return FM_OK;
    }
  }
  return fail(nullptr, FM_ERR_INVALID_ARG, std::string("unknown buffer name: ") + name);
}

int fm_trace_size(const fm_policy* p, size_t* bytes) {
  if (!p || !bytes) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL argument");
  *bytes = trace_record_bytes(p) * p->cfg.S * p->cfg.L;
  return FM_OK;
}

int fm_decode_trace(fm_policy* p, const float* noise, float* actions, void* trace, size_t bytes, void* stream) {
  if (!p || !actions || !trace) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  size_t need = 0;
  fm_trace_size(p, &need);
  if (bytes < need) return fail(p, FM_ERR_WORKSPACE, "trace buffer too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* a = p->at<float>(p->ly.a);
  if (noise && noise != a) FM_CUDA(p, cudaMemcpyAsync(a, noise, p->ly.a_bytes, cudaMemcpyDeviceToDevice, s));
  Trace tr;
  tr.base = static_cast<uint8_t*>(trace);
  tr.st = s;
  FM_CUDA(p, enqueue_decision(p, s, &tr));
  if (actions != a) FM_CUDA(p, cudaMemcpyAsync(actions, a, p->ly.a_bytes, cudaMemcpyDeviceToDevice, s));
  p->have_prev = true;
  FM_CUDA(p, cudaStreamSynchronize(s));
  if (tr.off != need) return fail(p, FM_ERR_INVALID_ARG, "internal: trace size mismatch");
  return FM_OK;
}

int fm_warm_trace_size(const fm_policy* p, size_t* bytes) {
  if (!p || !bytes) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL argument");
  *bytes = p->ly.a_bytes + trace_record_bytes(p) * p->cfg.L;
  return FM_OK;
}

int fm_decode_warm_trace(fm_policy* p, const float* noise, int executed, float* actions, void* trace, size_t bytes,
                         void* stream) {
  if (!p || !noise || !actions || !trace) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  const fm_config& c = p->cfg;
  if (!(c.warm_t > 0.f)) return fail(p, FM_ERR_UNSUPPORTED, "the policy was created with warm_t = 0");
  if (executed < 0 || executed > c.M) return fail(p, FM_ERR_INVALID_ARG, "executed must lie in [0, M]");
  if (!p->have_prev) return fail(p, FM_ERR_INVALID_ARG, "no previous chunk to warm-start from");
  size_t need = 0;
  fm_warm_trace_size(p, &need);
  if (bytes < need) return fail(p, FM_ERR_WORKSPACE, "trace buffer too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* a = p->at<float>(p->ly.a);
  float* prev = p->at<float>(p->ly.prev);
  FM_CUDA(p, cudaMemcpyAsync(prev, a, p->ly.a_bytes, cudaMemcpyDeviceToDevice, s));
  FM_CUDA(p, fm::warm_mix_launch(a, prev, noise, c.M, c.A, executed, c.warm_t, s));
  Trace tr;
  tr.base = static_cast<uint8_t*>(trace);
  tr.st = s;
  FM_CUDA(p, tr.rec(a, p->ly.a_bytes));   // a_tau, the input of the single Euler step
  FM_CUDA(p, enqueue_warm_traced(p, s, &tr));
  if (actions != a) FM_CUDA(p, cudaMemcpyAsync(actions, a, p->ly.a_bytes, cudaMemcpyDeviceToDevice, s));
  ++p->decisions;
  FM_CUDA(p, cudaStreamSynchronize(s));
  if (tr.off != need) return fail(p, FM_ERR_INVALID_ARG, "internal: trace size mismatch");
  return FM_OK;
}

int fm_test_launch_kernel(fm_policy* p, int layer, int step, int index, void* stream) {
  if (!p) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL policy");
  const fm_config& c = p->cfg;
  if (layer < 0 || layer >= c.L || step < 0 || step >= c.S || index < 0 || index >= p->dv.kernels_per_layer())
    return fail(p, FM_ERR_INVALID_ARG, "layer, step or kernel index out of range");
  LaunchOpts o;
  o.stream = static_cast<cudaStream_t>(stream);
  o.pdl = (c.flags & FM_FLAG_USE_PDL) != 0;   // as the decision launches it
  int seq = 0;
  o.seq = &seq;
  o.only = index;
  FM_CUDA(p, enqueue_layer(p, layer, step, layer == c.L - 1, o));
  if (seq <= index) return fail(p, FM_ERR_INVALID_ARG, "kernel index beyond this layer-step's launches");
  return FM_OK;
}

int fm_decode_timeline(fm_policy* p, const float* noise, float* actions, void* buf, size_t bytes, void* stream) {
  if (!p || !noise || !actions || !buf) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  if (bytes < 192 || reinterpret_cast<uintptr_t>(buf) % 16) return fail(p, FM_ERR_WORKSPACE, "buffer too small or unaligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long* tl = static_cast<unsigned long long*>(buf);
  const unsigned hdr[2] = {0u, static_cast<unsigned>(std::min<size_t>((bytes - 64) / 128, 0xffffffffu))};
  float* a = p->at<float>(p->ly.a);
  // the same plan as decode_actions, captured with the timeline buffer in its kernels'
  // parameters (a graph when the policy replays one, else launched one by one)
  cudaGraph_t g = nullptr;
  cudaGraphExec_t ge = nullptr;
  const bool use_graph = (p->cfg.flags & FM_FLAG_USE_GRAPH) != 0;
  if (use_graph) {
    FM_CUDA(p, cudaStreamBeginCapture(p->cap_stream, cudaStreamCaptureModeThreadLocal));
    cudaError_t e = enqueue_decision(p, p->cap_stream, nullptr, tl);
    cudaError_t e2 = cudaStreamEndCapture(p->cap_stream, &g);
    if (e != cudaSuccess || e2 != cudaSuccess) {
      if (g) cudaGraphDestroy(g);
      return cuda_fail(p, e != cudaSuccess ? e : e2, "capturing the timeline decision");
    }
    e = cudaGraphInstantiate(&ge, g, 0);
    if (e == cudaSuccess) e = cudaGraphUpload(ge, s);
    if (e != cudaSuccess) {
      cudaGraphDestroy(g);
      return cuda_fail(p, e, "instantiating the timeline decision");
    }
  }
  cudaError_t e = cudaSuccess;
  for (int pass = 0; pass < 2 && e == cudaSuccess; ++pass) {   // the first pass warms up
    e = cudaMemcpyAsync(tl, hdr, sizeof hdr, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && noise != a) e = cudaMemcpyAsync(a, noise, p->ly.a_bytes, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = use_graph ? cudaGraphLaunch(ge, s) : enqueue_decision(p, s, nullptr, tl);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e == cudaSuccess && actions != a) e = cudaMemcpyAsync(actions, a, p->ly.a_bytes, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (ge) cudaGraphExecDestroy(ge);
  if (g) cudaGraphDestroy(g);
  if (e != cudaSuccess) return cuda_fail(p, e, "timeline decision");
  p->have_prev = true;
  return FM_OK;
}

int fm_test_kernel_count(const fm_policy* p, int* per_layer, int* per_decision) {
  if (!p || !per_layer || !per_decision) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL argument");
  *per_layer = p->dv.kernels_per_layer();
  *per_decision = 1 + p->cfg.S * p->cfg.L * p->dv.kernels_per_layer() + (p->dv.rowfuse ? p->cfg.S : 0);
  return FM_OK;
}

int fm_test_attn_plan(const fm_policy* p, int* keys_per_slice, int* slices) {
  if (!p || !keys_per_slice || !slices) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL argument");
  *keys_per_slice = p->dv.attn_kc;
  *slices = p->dv.attn_nsplit;
  return FM_OK;
}

int fm_test_quant_e4m3(const float* x, int64_t n, float scale, uint8_t* codes, void* stream) {
  if (!x || !codes || n < 0) return fail(nullptr, FM_ERR_INVALID_ARG, "bad argument");
  if (!(scale > 0.f)) return fail(nullptr, FM_ERR_INVALID_ARG, "scale must be positive");
  const cudaError_t e = fm::quant_e4m3_launch(x, n, scale, codes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FM_OK : cuda_fail(nullptr, e, "quant_e4m3");
}

int fm_packed_weight_bytes(int N, int K, int fmt, size_t* bytes) {
  if (!bytes) return fail(nullptr, FM_ERR_INVALID_ARG, "bytes is NULL");
  if (N <= 0 || K <= 0 || N % 128 || K % 128) return fail(nullptr, FM_ERR_SHAPE, "N, K must be multiples of 128");
  if (fmt != FM_FMT_FP8 && fmt != FM_FMT_BF16 && fmt != FM_FMT_NVFP4)
    return fail(nullptr, FM_ERR_UNSUPPORTED, "format");
  *bytes = fm::packed_weight_bytes(N, K, fmt);
  return FM_OK;
}

int fm_pack_weight(const float* w, const float* gamma, int N, int K, int fmt, void* packed, float* scale_out,
                   void* stream) {
  if (!w || !packed || !scale_out) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL argument");
  if (N <= 0 || K <= 0 || N % 128 || K % 128) return fail(nullptr, FM_ERR_SHAPE, "N, K must be multiples of 128");
  if (fmt != FM_FMT_FP8 && fmt != FM_FMT_BF16 && fmt != FM_FMT_NVFP4)
    return fail(nullptr, FM_ERR_UNSUPPORTED, "format");
  if (reinterpret_cast<uintptr_t>(packed) % kAlign) return fail(nullptr, FM_ERR_ALIGN, "packed not 1024-aligned");
  // The caller's 4-byte scale slot doubles as the amax accumulator: the amax kernel
  // fills it, then one thread reads it and overwrites it with the scale.
  const cudaError_t e = fm::pack_weight(w, gamma, N, K, fmt, packed, scale_out,
                                        reinterpret_cast<unsigned*>(scale_out), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FM_OK : cuda_fail(nullptr, e, "pack_weight");
}

int fm_test_skinny_gemm_tile(const void* a, int M, int K, const void* w_packed, int N, int fmt, int s,
                             int cluster_reduce, int tile_rows, float* partials, void* stream);

int fm_test_skinny_gemm(const void* a, int M, int K, const void* w_packed, int N, int fmt, int s, int cluster_reduce,
                        float* partials, void* stream) {
  return fm_test_skinny_gemm_tile(a, M, K, w_packed, N, fmt, s, cluster_reduce, 128, partials, stream);
}

int fm_test_skinny_gemm_tile(const void* a, int M, int K, const void* w_packed, int N, int fmt, int s,
                             int cluster_reduce, int tile_rows, float* partials, void* stream) {
  if (!a || !w_packed || !partials) return fail(nullptr, FM_ERR_INVALID_ARG, "NULL argument");
  if (fmt != FM_FMT_FP8 && fmt != FM_FMT_BF16 && fmt != FM_FMT_NVFP4)
    return fail(nullptr, FM_ERR_UNSUPPORTED, "format");
  if (!aligned16(a) || reinterpret_cast<uintptr_t>(w_packed) % kAlign)
    return fail(nullptr, FM_ERR_ALIGN, "a must be 16-byte and w_packed 1024-byte aligned");
  if (fmt == FM_FMT_NVFP4) {
    if (cluster_reduce != 1 || tile_rows != 128)
      return fail(nullptr, FM_ERR_SHAPE, "NVFP4 GEMM writes every slice of 128-row tiles: cluster_reduce 1, tile 128");
    fm::Nvfp4Shape g;
    if (fm::nvfp4_plan(M, N, K, s, &g) != FM_OK)
      return fail(nullptr, FM_ERR_SHAPE, "GEMM shape/split precondition violated");
    CUtensorMap ta;
    if (!fm::nvfp4_tmap_act(&ta, a, g)) return fail(nullptr, FM_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    cudaError_t e = fm::nvfp4_configure();
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "nvfp4_configure");
    int* err_word = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&err_word), fm_standalone_err);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "error word");
    LaunchOpts o;
    o.stream = static_cast<cudaStream_t>(stream);
    e = fm::nvfp4_gemm_launch(ta, w_packed, g, partials, nullptr, nullptr, nullptr, nullptr, err_word, o);
    return e == cudaSuccess ? FM_OK : cuda_fail(nullptr, e, "nvfp4 gemm launch");
  }
  fm::GemmShape g;
  const int st = fm::gemm_plan(M, N, K, fmt == FM_FMT_FP8, s, cluster_reduce, &g, tile_rows);
  if (st != FM_OK) return fail(nullptr, st, "GEMM shape/split precondition violated");
  CUtensorMap ta;
  if (!fm::gemm_tmap_act(&ta, a, g))
    return fail(nullptr, FM_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  cudaError_t e = fm::gemm_configure();
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "gemm_configure");
  int* err_word = nullptr;   // looked up per call: the address is per device
  e = cudaGetSymbolAddress(reinterpret_cast<void**>(&err_word), fm_standalone_err);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "error word");
  LaunchOpts o;
  o.stream = static_cast<cudaStream_t>(stream);
  e = fm::gemm_launch(w_packed, ta, g, partials, err_word, o);
  return e == cudaSuccess ? FM_OK : cuda_fail(nullptr, e, "skinny_gemm launch");
}

int fm_gemm_consumer_scratch_bytes(int M, int N, int K, int fmt, int s, size_t* bytes) {
  if (!bytes) return fail(nullptr, FM_ERR_INVALID_ARG, "bytes is NULL");
  const char* why = "";
  const int st = fm::gemm_consumer_scratch_bytes(M, N, K, fmt, s, bytes, &why);
  return st == FM_OK ? FM_OK : fail(nullptr, st, why);
}

int fm_gemm_consumer(const void* a, int M, int K, const void* w_packed, int N, int fmt, int s, const float* s_a,
                     const float* s_w, const float* bias, float* x, const float* gate, const float* scale,
                     const float* shift, float eps, const float* s_q, void* q, void* scratch, size_t scratch_bytes,
                     void* stream) {
  int* err_word = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&err_word), fm_standalone_err);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "error word");
  const fm::GemmConsumerArgs g{a, M, K, N, fmt, s, w_packed, s_a, s_w, bias, x, gate, scale, shift, eps, s_q, q};
  const char* why = "";
  const int st = fm::gemm_consumer_run(g, static_cast<float*>(scratch), scratch_bytes, err_word,
                                       static_cast<cudaStream_t>(stream), &why);
  return st == FM_OK ? FM_OK : fail(nullptr, st, why);
}

int fm_test_consumer(const float* partials, int nparts, int M, int N, const float* s_a, const float* s_w,
                     const float* bias, float* x, const float* gate, const float* scale, const float* shift, float eps,
                     const float* s_q, void* q, int act_fmt, void* stream) {
  if (!partials || !s_a || !s_w || !x || !gate || !scale || !shift || !s_q || !q)
    return fail(nullptr, FM_ERR_INVALID_ARG, "NULL argument");
  if (nparts < 1 || M < 1 || N < 4 || N % 4 || N > 16384) return fail(nullptr, FM_ERR_SHAPE, "bad shape");
  if (act_fmt != FM_FMT_FP8 && act_fmt != FM_FMT_BF16) return fail(nullptr, FM_ERR_INVALID_ARG, "act_fmt");
  const void* ptrs[7] = {partials, x, gate, scale, shift, q, bias ? bias : partials};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return fail(nullptr, FM_ERR_ALIGN, "pointers must be 16-byte aligned");
  fm::RowArgs r = {};
  r.M = M;
  r.N = N;
  r.parts = partials;
  r.nparts = nparts;
  r.sa = s_a;
  r.sw = s_w;
  r.bias = bias;
  r.gate = gate;
  r.x = x;
  r.do_quant = 1;
  r.scale = scale;
  r.shift = shift;
  r.sq = s_q;
  r.q = q;
  r.q_fp8 = act_fmt == FM_FMT_FP8;
  r.eps = eps;
  LaunchOpts o;
  o.stream = static_cast<cudaStream_t>(stream);
  const cudaError_t e = fm::row_launch(r, o);
  return e == cudaSuccess ? FM_OK : cuda_fail(nullptr, e, "consumer launch");
}

int fm_test_layer(fm_policy* p, const float* x_in, int layer, int step, float* x_out, void* q_out, void* stream) {
  if (!p || !x_in || !x_out || !q_out) return fail(p, FM_ERR_INVALID_ARG, "NULL argument");
  if (layer < 0 || layer >= p->cfg.L || step < 0 || step >= p->cfg.S) return fail(p, FM_ERR_SHAPE, "bad layer/step");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LaunchOpts o;
  o.stream = s;
  o.pdl = (p->cfg.flags & FM_FLAG_USE_PDL) != 0;
  fm::RowArgs r = {};
  r.M = p->cfg.M;
  r.N = p->cfg.d;
  r.x = p->at<float>(p->ly.x);
  r.x_src = x_in;
  r.do_quant = 1;
  r.scale = p->mod(step, layer, 0);
  r.shift = p->mod(step, layer, 1);
  r.sq = p->ascale(layer, FM_SITE_ATTN_IN);
  r.q = p->at<void>(p->ly.q);
  r.q_fp8 = p->dv.q_store;
  r.eps = p->cfg.rms_eps;
  if (p->dv.rowfuse) {   // the QKV GEMM normalises x itself: hand it the row sums instead
    r.do_quant = 0;
    r.ssq = p->at<float>(p->ly.ssq);
    r.ssq_tiles = p->cfg.d / 128;
  }
  FM_CUDA(p, fm::row_launch(r, o));
  FM_CUDA(p, enqueue_layer(p, layer, step, false, o));
  if (p->dv.rowfuse) {   // the next layer's pre-attention operand, as a separate consumer computes it
    fm::RowArgs n = {};
    const int ln = (layer + 1) % p->cfg.L;
    n.M = p->cfg.M;
    n.N = p->cfg.d;
    n.x = p->at<float>(p->ly.x);
    n.do_quant = 1;
    n.scale = p->mod(step, ln, 0);
    n.shift = p->mod(step, ln, 1);
    n.sq = p->ascale(ln, FM_SITE_ATTN_IN);
    n.q = p->at<void>(p->ly.q);
    n.q_fp8 = p->dv.q_store;
    n.eps = p->cfg.rms_eps;
    FM_CUDA(p, fm::row_launch(n, o));
  }
  const size_t xb = static_cast<size_t>(p->cfg.M) * p->cfg.d * 4;
  FM_CUDA(p, cudaMemcpyAsync(x_out, p->at<void>(p->ly.x), xb, cudaMemcpyDeviceToDevice, s));
  FM_CUDA(p, cudaMemcpyAsync(q_out, p->at<void>(p->ly.q), static_cast<size_t>(p->cfg.M) * p->cfg.d * p->dv.act_bytes,
                             cudaMemcpyDeviceToDevice, s));
  return FM_OK;
}

}  // extern "C"
