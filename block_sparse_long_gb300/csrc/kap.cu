// Kernel-Aware Proxy (KAP): computation-order mask from stride-sampled queries and keys.
//
// CoSA (arXiv 2607.25291) Sec. 4.2, Eqs. (8)-(14), Algorithm A lines 2-5.  For each
// request and query head, with sampled rows r (positions r*s) and keys c (positions c*s):
//   logits  l[r,c] = q~_r . k~_c * scale for causal (c <= r), existing keys;
//   Eq. (9)-(10) reduce, for the row softmax of Eq. (8), to
//           Pbar[r,j] = exp(bm[r,j] - M_r), bm = max of l over the sampled keys of block j,
//           M_r = max_j bm[r,j]  (the softmax normaliser cancels in the max-normalisation);
//   Eq. (11) s_ij = sum over the sampled rows of query block i of Pbar[r,j];
//   Eq. (12) h_ij = 1 iff some row of block i attains its maximum in block j;
//   Eq. (13) rho_i = HRM blocks by descending score, then the rest (ties: lower ID first);
//   Eq. (14) M_KAP[i, 0:K_i] = rho_i[0:K_i], K_i = ceil(B1 * (i+1)).
//
// Exactness.  The logits run on tcgen05 tensor cores in fp32; every decision that fp32 could
// get wrong is settled in float64:
//   pass 1 (kap_logits<ROWMAX>)  per row: the four largest fp32 logits and their keys;
//   kap_exact                    per row: error bound e_r >= |fp32 logit - exact logit| for every
//                                 key of the row (from ||q_r|| * max ||k|| and the accumulation
//                                 length); if the runner-up is more than 2 e_r below the maximum
//                                 the argmax key is certain and M_r is its float64 logit;
//                                 otherwise every key within 2 e_r is re-evaluated in float64;
//                                 the HRM blocks of the row follow exactly;
//   pass 2 (kap_logits<SCORES>)  per (query block, key block): fp32 score and a rigorous bound
//                                 on its error, given the float64 M_r;
//   kap_select                   flag-grouped sort of the fp32 scores; every adjacent pair whose
//                                 order, and the budget cut, that the bounds cannot certify is
//                                 recomputed with float64 logits and exp, and re-sorted.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

// Fixed scratch for callers that cannot allocate device memory (cosa_proxy_select_static).
// Every GPU that loads this library holds it until the process exits; all calls share it.
__device__ __align__(256) uint8_t cosa_kap_static_scratch[cosa::kStaticScratchBytes];

namespace cosa {
namespace {

constexpr int kRowTile = 128;           // sampled rows per CTA of the logits kernel
constexpr int kKeyTile = 128;           // sampled keys per UMMA
constexpr int kSelectThreads = 256;
// |fp32 logit - exact| <= kKappa * ||q|| * ||k|| * scale for d <= 128.  The products of bf16
// inputs are exact in fp32; summing them in groups of at most 16 aligned to the group's largest
// term and truncated to fp32 width, then adding each group to a truncating fp32 accumulator,
// loses at most (16 + 8) * 2^-23 = 48 * 2^-24 of sum |q_k k_k| <= ||q|| ||k||.  kKappa = 64 * 2^-24
// covers that model; on GB300 the largest error measured over normal, Student-t, mixed-magnitude
// and one-large-many-small inputs was 13 * 2^-24 of sum |q_k k_k|.  The CUDA-core fp32 dot
// products (4 sequential FMAs per lane, a 5-level shuffle tree) stay within 9 * 2^-24.
constexpr float kKappa = 1.0f / 262144.0f;
constexpr int kTop = 4;                 // candidates per row kept by the row-max pass

struct KapArgs {
  const uint16_t* q;
  const int32_t* cu_seqlens;
  const uint16_t* k_cache;
  const int32_t* page_table;
  int32_t* mask;
  int32_t* mask_len;
  int32_t* status;
  // workspace
  int64_t* row_off;      // [B+1]: first sampled-row record of request b (times Hq)
  int64_t* sc_off;       // [B+1]: first score of request b (times Hq)
  float* knorm;          // [B * Hkv]: max ||k~|| of the request's existing sampled keys
  float* kbnorm;         // [B * Hkv * nqb_max]: max ||k~|| over the sampled keys of each block
  float* topv;           // per sampled row: kTop largest fp32 logits (scaled, descending), -inf pad
  int32_t* topc;         // per sampled row: their key indices
  float* qnorm;          // per sampled row: ||q~_r|| rounded up
  double* M;             // per sampled row: exact maximum logit (scaled), -inf if none
  float* err;            // per sampled row: error bound e_r of its fp32 logits (scaled)
  int32_t* rflags;       // per sampled row: bit 0 = several HRM candidates (bitmap valid), bit 1 = empty
  int32_t* c1;           // per sampled row: the exact argmax key (the first one if several tie)
  uint32_t* hrm_bits;    // per sampled row: bitmap of HRM blocks, words_per_row words (ambiguous rows only)
  float* score;          // per (request, head): nqb x nqb fp32 scores, row i = query block
  float* score_err;      // same shape: bound on |score - exact score|
  int num_reqs, num_q_heads, num_kv_heads, head_dim, block_size, page_size, stride, kb;
  int total_tokens, max_seqlen, num_pages, max_pages_per_req, mask_pitch, budget_ppm;
  int nqb_max, nrow_tiles_max, words_per_row;
  double sm_scale;
};

struct ReqInfo {
  int tok0, L, R, nqb, req_pages;
  bool ok;
};

__device__ __forceinline__ ReqInfo req_info(const KapArgs& a, int b) {
  ReqInfo r;
  r.tok0 = a.cu_seqlens[b];
  r.L = a.cu_seqlens[b + 1] - r.tok0;
  r.ok = !(r.L < 0 || r.L > a.max_seqlen || r.tok0 < 0 || r.tok0 + r.L > a.total_tokens);
  if (!r.ok) r.L = 0;
  r.R = (r.L + a.stride - 1) / a.stride;
  r.nqb = (r.L + a.block_size - 1) / a.block_size;
  r.req_pages = (r.L + a.page_size - 1) / a.page_size;
  return r;
}

// Address of sampled key c of request b, kv head kvh, or nullptr if its page does not exist.
__device__ __forceinline__ const uint16_t* key_ptr(const KapArgs& a, const ReqInfo& ri, int b, int kvh, int c) {
  if (c < 0 || c >= ri.R) return nullptr;
  const int pos = c * a.stride;
  const int p = pos / a.page_size;
  if (p >= ri.req_pages) return nullptr;
  const int phys = a.page_table[static_cast<size_t>(b) * a.max_pages_per_req + p];
  if (phys < 0 || phys >= a.num_pages) return nullptr;
  const int off = pos - p * a.page_size;
  return a.k_cache + ((static_cast<size_t>(phys) * a.page_size + off) * a.num_kv_heads + kvh) * a.head_dim;
}

__device__ __forceinline__ const uint16_t* query_ptr(const KapArgs& a, const ReqInfo& ri, int h, int r) {
  return a.q + ((static_cast<size_t>(ri.tok0) + static_cast<size_t>(r) * a.stride) * a.num_q_heads + h) * a.head_dim;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); }

// 16-byte async copy; with valid == false nothing is read and the destination is zero-filled
// (`fallback` is any mapped global address, passed so the operand is never null).
__device__ __forceinline__ void cp_async_16(void* dst, const void* src, bool valid, const void* fallback) {
  const uint32_t n = valid ? 16u : 0u;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(valid ? src : fallback),
               "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// warp dot products over d (lanes split d into contiguous slices)
template <int HD>
__device__ __forceinline__ float warp_dot_f32(const uint16_t* x, const uint16_t* y) {
  constexpr int PER = HD / 32;
  const int l = threadIdx.x & 31;
  float acc = 0.0f;
#pragma unroll
  for (int e = 0; e < PER; ++e) acc = fmaf(bf16_to_f32(x[l * PER + e]), bf16_to_f32(y[l * PER + e]), acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

template <int HD>
__device__ __forceinline__ double warp_dot_f64(const uint16_t* x, const uint16_t* y) {
  constexpr int PER = HD / 32;
  const int l = threadIdx.x & 31;
  double acc = 0.0;
#pragma unroll
  for (int e = 0; e < PER; ++e)
    acc = fma(static_cast<double>(bf16_to_f32(x[l * PER + e])), static_cast<double>(bf16_to_f32(y[l * PER + e])), acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

// ---------------------------------------------------------------------------
// setup: per-request offsets into the workspace, zeroed key norms, input checks
// ---------------------------------------------------------------------------
__global__ void kap_setup_kernel(KapArgs a) {
  if (threadIdx.x == 0) {
    int64_t ro = 0, so = 0;
    for (int b = 0; b < a.num_reqs; ++b) {
      a.row_off[b] = ro;
      a.sc_off[b] = so;
      const ReqInfo ri = req_info(a, b);
      if (!ri.ok) report_status(a.status, kStatusBadInput);
      ro += static_cast<int64_t>(a.num_q_heads) * ri.R;
      so += static_cast<int64_t>(a.num_q_heads) * ri.nqb * ri.nqb;
    }
    a.row_off[a.num_reqs] = ro;
    a.sc_off[a.num_reqs] = so;
  }
  for (int e = threadIdx.x; e < a.num_reqs * a.num_kv_heads; e += blockDim.x) a.knorm[e] = 0.0f;
  for (int e = threadIdx.x; e < a.num_reqs * a.num_kv_heads * a.nqb_max; e += blockDim.x) a.kbnorm[e] = 0.0f;
}

// max ||k~_c|| over the existing sampled keys of (request, kv head); rounded up
template <int HD>
__global__ void kap_knorm_kernel(KapArgs a) {
  const int b = blockIdx.y / a.num_kv_heads, kvh = blockIdx.y % a.num_kv_heads;
  const ReqInfo ri = req_info(a, b);
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const uint16_t* k = key_ptr(a, ri, b, kvh, c);
  float n = 0.0f;
  if (k != nullptr) {
    float s2 = 0.0f;
    for (int e = 0; e < HD; ++e) {
      const float x = bf16_to_f32(k[e]);
      s2 = fmaf(x, x, s2);
    }
    n = sqrtf(s2) * (1.0f + 1.0f / 65536.0f);
  }
  if (n > 0.0f) {
    const int j = (c * a.stride) / a.block_size;
    atomicMax(reinterpret_cast<int*>(&a.kbnorm[(static_cast<size_t>(b) * a.num_kv_heads + kvh) * a.nqb_max + j]),
              __float_as_int(n));
  }
  for (int o = 16; o > 0; o >>= 1) n = fmaxf(n, __shfl_xor_sync(0xffffffffu, n, o));
  if ((threadIdx.x & 31) == 0 && n > 0.0f)
    atomicMax(reinterpret_cast<int*>(&a.knorm[b * a.num_kv_heads + kvh]), __float_as_int(n));
}

// ---------------------------------------------------------------------------
// sampled logits on tcgen05: 128 sampled rows x all causal sampled keys
// ---------------------------------------------------------------------------
enum { kModeRowMax = 0, kModeScores = 1 };

template <int HD>
struct alignas(1024) KapTileSmem {
  uint8_t q[kRowTile * HD * 2];        // [HD/64][128][128 B] SW128
  uint8_t k[2][kKeyTile * HD * 2];
  uint32_t kvalid[2][kKeyTile / 32];
  uint64_t bar[2];
  uint32_t tmem_base;
  int32_t abort_flag;
};

template <int HD>
__device__ __forceinline__ void load_rows_sw128(uint8_t* dst, const uint16_t* src, bool valid, int row,
                                                const void* fallback) {
  // one 128-element (or 64-element) row: HD/8 chunks of 16 B into the SW128 layout
#pragma unroll
  for (int c16 = 0; c16 < HD / 8; ++c16) {
    const int half = c16 >> 3, ch = c16 & 7;
    cp_async_16(dst + half * (128 * 128) + sw128_offset(row, ch), valid ? src + c16 * 8 : nullptr, valid, fallback);
  }
}

template <int HD, int KB, int MODE>
__global__ void __launch_bounds__(128) kap_logits_kernel(KapArgs a) {
  using S = KapTileSmem<HD>;
  extern __shared__ uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int idx = blockIdx.x;
  const int h = idx % a.num_q_heads;
  idx /= a.num_q_heads;
  const int b = idx % a.num_reqs;
  const int rt = a.nrow_tiles_max - 1 - idx / a.num_reqs;  // heaviest row tiles first
  const ReqInfo ri = req_info(a, b);
  if (rt * kRowTile >= ri.R) return;
  const int kvh = h / (a.num_q_heads / a.num_kv_heads);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int r = rt * kRowTile + t;              // this thread's sampled row
  const bool row_ok = r < ri.R;
  const int64_t rec = a.row_off[b] + static_cast<int64_t>(h) * ri.R + r;
  const int nkt = rt + 1;                       // causal key tiles
  const float scale = static_cast<float>(a.sm_scale);

  if (t == 0) {
    mbar_init(&sm.bar[0], 1);
    mbar_init(&sm.bar[1], 1);
    sm.abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, 256);
    tmem_relinquish();
  }
  // Q~ tile and key tile 0
  load_rows_sw128<HD>(sm.q, row_ok ? query_ptr(a, ri, h, r) : nullptr, row_ok, t, a.q);
  auto load_keys = [&](int kt, int buf) {
    const int c = kt * kKeyTile + t;
    const uint16_t* kp = key_ptr(a, ri, b, kvh, c);
    load_rows_sw128<HD>(sm.k[buf], kp, kp != nullptr, t, a.q);
    const unsigned bal = __ballot_sync(0xffffffffu, kp != nullptr);
    if (lane == 0) sm.kvalid[buf][warp] = bal;
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  load_keys(0, 0);
  cp_async_wait_all();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  constexpr uint32_t idesc = idesc_bf16_f32(128, kKeyTile, false, false);
  auto issue = [&](int buf) {
    if (t == 0) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint64_t ad = smem_desc_sw128(smem_u32(&sm.q[(kk >> 2) * 128 * 128 + (kk & 3) * 32]), 16, 1024);
        const uint64_t bd = smem_desc_sw128(smem_u32(&sm.k[buf][(kk >> 2) * 128 * 128 + (kk & 3) * 32]), 16, 1024);
        umma_ss(tmem + buf * 128, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
      umma_commit(&sm.bar[buf]);
    }
  };
  issue(0);
  if (nkt > 1) load_keys(1, 1);

  // per-row state
  float topv[kTop];                             // kTop largest raw fp32 logits, descending
  int topc[kTop];
#pragma unroll
  for (int m = 0; m < kTop; ++m) { topv[m] = -INFINITY; topc[m] = -1; }
  float M32 = -INFINITY, ebase = 0.0f;
  int64_t sbase = 0;
  int nqb = ri.nqb;
  const float* kbn = a.kbnorm + (static_cast<size_t>(b) * a.num_kv_heads + kvh) * a.nqb_max;
  if (MODE == kModeScores) {
    if (row_ok) {
      M32 = static_cast<float>(a.M[rec]);
      ebase = kKappa * scale * a.qnorm[rec] * 1.001f;
    }
    sbase = a.sc_off[b] + static_cast<int64_t>(h) * nqb * nqb;
  }
  const int qblk = r / KB;                      // query block of this row
  bool ok = true;
  for (int kt = 0; kt < nkt; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nkt) {                         // key tile kt+1 has landed: start its UMMA
      cp_async_wait_all();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      issue(buf ^ 1);
    }
    // the whole CTA agrees on the outcome, so every thread leaves the loop together
    ok = __syncthreads_and(wait_parity_bounded(&sm.bar[buf], (kt >> 1) & 1, &sm.abort_flag, a.status)) != 0;
    if (!ok) break;
    tc_fence_after();
    uint32_t kvalid[kKeyTile / 32];
#pragma unroll
    for (int w = 0; w < kKeyTile / 32; ++w) kvalid[w] = sm.kvalid[buf][w];
    __syncthreads();                            // buffer `buf` is free: UMMA kt is done, flags copied
    if (kt + 2 < nkt) load_keys(kt + 2, buf);
    // epilogue of key tile kt
    const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16) + buf * 128;
    const int last_col = r - kt * kKeyTile;     // causal: columns <= last_col
#pragma unroll
    for (int cc = 0; cc < kKeyTile / 32; ++cc) {
      uint32_t rv[32];
      tmem_ld32(taddr + cc * 32, rv);
      tmem_wait_ld();
      const uint32_t vbits = kvalid[cc];
      if (MODE == kModeRowMax) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = cc * 32 + e;
          if (!row_ok || col > last_col || !((vbits >> e) & 1u)) continue;
          const float x = __uint_as_float(rv[e]);
          if (x > topv[3]) {                    // insertion into the sorted top-4 (ties keep the first)
            const int key = kt * kKeyTile + col;
            if (x > topv[2]) {
              topv[3] = topv[2]; topc[3] = topc[2];
              if (x > topv[1]) {
                topv[2] = topv[1]; topc[2] = topc[1];
                if (x > topv[0]) {
                  topv[1] = topv[0]; topc[1] = topc[0]; topv[0] = x; topc[0] = key;
                } else {
                  topv[1] = x; topc[1] = key;
                }
              } else {
                topv[2] = x; topc[2] = key;
              }
            } else {
              topv[3] = x; topc[3] = key;
            }
          }
        }
      } else {
#pragma unroll
        for (int g = 0; g < 32 / KB; ++g) {
          float bm = -INFINITY;
#pragma unroll
          for (int e = g * KB; e < (g + 1) * KB; ++e) {
            const int col = cc * 32 + e;
            if (row_ok && col <= last_col && ((vbits >> e) & 1u)) bm = fmaxf(bm, __uint_as_float(rv[e]));
          }
          const int j = kt * (kKeyTile / KB) + cc * (32 / KB) + g;
          float x = 0.0f, xe = 0.0f;
          if (bm != -INFINITY && M32 != -INFINITY) {
            const float u = fmaf(bm, scale, -M32);
            x = expf(u);
            // |u - exact| <= kappa * scale * ||q|| * (largest ||k|| of block j) plus the rounding of
            // the scaled logit, of M_r and of the subtraction; expf adds at most 2 ulp; a value
            // below exp(-80) is only bounded absolutely
            const float du = ebase * __ldg(kbn + j) + 1.2e-7f * (2.0f * fabsf(M32) + fabsf(u) + 1.0f);
            xe = x * (expm1f(du) * 1.01f + 3.0e-7f) + ((u < -80.0f) ? 2.0e-35f : 0.0f);
          }
#pragma unroll
          for (int o = KB / 2; o > 0; o >>= 1) {
            x += __shfl_xor_sync(0xffffffffu, x, o);
            xe += __shfl_xor_sync(0xffffffffu, xe, o);
          }
          if ((lane % KB) == 0 && qblk < nqb && j <= qblk) {
            const int64_t o = sbase + static_cast<int64_t>(qblk) * nqb + j;
            a.score[o] = x;
            a.score_err[o] = xe + x * (4.0f * 6.0e-8f);   // rounding of the kb-term sum
          }
        }
      }
    }
    tc_fence_before();
  }
  if (MODE == kModeRowMax && row_ok) {
#pragma unroll
    for (int m = 0; m < kTop; ++m) {
      a.topv[rec * kTop + m] = (topv[m] == -INFINITY) ? -INFINITY : topv[m] * scale;
      a.topc[rec * kTop + m] = topc[m];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------------------
// exact row maxima (float64) and HRM blocks of each sampled row; one warp per row
// ---------------------------------------------------------------------------
template <int HD>
__global__ void __launch_bounds__(256) kap_exact_kernel(KapArgs a) {
  const int warps_per_cta = blockDim.x / 32;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * warps_per_cta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  // locate (b, h, r) of record gw
  const int64_t total = a.row_off[a.num_reqs];
  if (gw >= total) return;
  int b = 0;
  while (b + 1 < a.num_reqs && a.row_off[b + 1] <= gw) ++b;
  const ReqInfo ri = req_info(a, b);
  const int64_t local = gw - a.row_off[b];
  const int h = static_cast<int>(local / ri.R);
  const int r = static_cast<int>(local % ri.R);
  const int kvh = h / (a.num_q_heads / a.num_kv_heads);
  const uint16_t* qr = query_ptr(a, ri, h, r);
  // ||q_r||
  float s2 = 0.0f;
  for (int e = lane; e < HD; e += 32) {
    const float x = bf16_to_f32(qr[e]);
    s2 = fmaf(x, x, s2);
  }
  for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
  const float qn = sqrtf(s2) * (1.0f + 1.0f / 65536.0f);
  // bound on |fp32 logit - exact| for every key of the row (largest key norm of the request)
  const float e_r = kKappa * static_cast<float>(a.sm_scale) * qn * a.knorm[b * a.num_kv_heads + kvh] * 1.001f + 1e-30f;
  const double scale = a.sm_scale;
  float tv[kTop];
  int tc[kTop];
#pragma unroll
  for (int m = 0; m < kTop; ++m) { tv[m] = a.topv[gw * kTop + m]; tc[m] = a.topc[gw * kTop + m]; }
  if (lane == 0) { a.qnorm[gw] = qn; a.err[gw] = e_r; }
  if (tv[0] == -INFINITY) {
    if (lane == 0) { a.M[gw] = -INFINITY; a.rflags[gw] = 2; a.c1[gw] = -1; }
    return;
  }
  // a key can hold the exact maximum only if its fp32 logit is within 2 e_r of the largest one
  const float window = tv[0] - 2.0f * e_r;
  if (tv[1] < window) {
    const double lx = warp_dot_f64<HD>(qr, key_ptr(a, ri, b, kvh, tc[0])) * scale;
    if (lane == 0) { a.M[gw] = lx; a.rflags[gw] = 0; a.c1[gw] = tc[0]; }
    return;
  }
  uint32_t* bits = a.hrm_bits + gw * a.words_per_row;
  for (int w = lane; w < a.words_per_row; w += 32) bits[w] = 0u;
  __syncwarp();
  double best = -INFINITY;
  int best_c = -1;
  if (tv[kTop - 1] < window) {
    // every candidate is among the kept top keys: evaluate them in float64
    double ex[kTop];
#pragma unroll
    for (int m = 0; m < kTop; ++m) {
      ex[m] = -INFINITY;
      if (tv[m] >= window) ex[m] = warp_dot_f64<HD>(qr, key_ptr(a, ri, b, kvh, tc[m])) * scale;
      if (ex[m] > best) { best = ex[m]; best_c = tc[m]; }
    }
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < kTop; ++m)
        if (ex[m] == best) {
          const int j = (tc[m] * a.stride) / a.block_size;
          bits[j >> 5] |= 1u << (j & 31);
        }
    }
  } else {
    // more near-ties than kept: scan the row; fp32 screen, float64 for the survivors
    const float thr = tv[0] - 3.0f * e_r;
    for (int c = 0; c <= r; ++c) {
      const uint16_t* kc = key_ptr(a, ri, b, kvh, c);
      if (kc == nullptr) continue;
      if (warp_dot_f32<HD>(qr, kc) * static_cast<float>(scale) < thr) continue;
      const double lx = warp_dot_f64<HD>(qr, kc) * scale;
      if (lx > best) { best = lx; best_c = c; }
    }
    for (int c = 0; c <= r; ++c) {
      const uint16_t* kc = key_ptr(a, ri, b, kvh, c);
      if (kc == nullptr) continue;
      if (warp_dot_f32<HD>(qr, kc) * static_cast<float>(scale) < thr) continue;
      if (warp_dot_f64<HD>(qr, kc) * scale == best && lane == 0) {
        const int j = (c * a.stride) / a.block_size;
        bits[j >> 5] |= 1u << (j & 31);
      }
    }
  }
  __syncwarp();
  if (lane == 0) { a.M[gw] = best; a.rflags[gw] = 1; a.c1[gw] = best_c; }
}

// ---------------------------------------------------------------------------
// per query block: flag-grouped sort, certification, float64 repair, mask row
// ---------------------------------------------------------------------------
// dynamic shared memory of kap_select for `cap` candidates (a power of two)
__host__ __device__ inline size_t select_smem_bytes(int cap) {
  return static_cast<size_t>(cap) * (8 + 4 + 4 + 4 + 4 + 8 + 1) + 64;
}

__device__ __forceinline__ unsigned long long sort_key(bool hrm, float s, int j) {
  // descending order of the key = HRM first, then score descending, then block ascending
  return (static_cast<unsigned long long>(hrm) << 63) | (static_cast<unsigned long long>(__float_as_uint(s)) << 31) |
         static_cast<unsigned long long>(0x7FFFFFFF - j);
}
__device__ __forceinline__ int key_block(unsigned long long k) { return 0x7FFFFFFF - static_cast<int>(k & 0x7FFFFFFFull); }

template <int HD>
__global__ void __launch_bounds__(kSelectThreads) kap_select_kernel(KapArgs a, int cap) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  unsigned long long* key = reinterpret_cast<unsigned long long*>(smem_raw);  // [cap] sort keys
  double* rep_val = reinterpret_cast<double*>(key + cap);                      // [cap] exact scores
  float* lo = reinterpret_cast<float*>(rep_val + cap);                         // [cap] lower bounds
  float* hi = lo + cap;                                                        // [cap] upper bounds
  float* suf = hi + cap;                                                       // [cap] suffix max of hi
  int32_t* rep_pos = reinterpret_cast<int32_t*>(suf + cap);                    // [cap] positions to repair
  uint8_t* hrm = reinterpret_cast<uint8_t*>(rep_pos + cap);                    // [cap] HRM flags
  __shared__ int32_t n_rep_s, n_hrm_s;

  const int tid = threadIdx.x;
  int idx = blockIdx.x;
  const int h = idx % a.num_q_heads;
  idx /= a.num_q_heads;
  const int b = idx % a.num_reqs;
  const int i = a.nqb_max - 1 - idx / a.num_reqs;
  const ReqInfo ri = req_info(a, b);
  const size_t mrow = (static_cast<size_t>(b) * a.num_q_heads + h) * a.nqb_max + i;
  int32_t* out = a.mask + mrow * a.mask_pitch;
  if (i >= ri.nqb) {
    for (int k = tid; k < a.mask_pitch; k += blockDim.x) out[k] = -1;
    if (tid == 0) a.mask_len[mrow] = 0;
    return;
  }
  const int J = i + 1;
  const int K = max(1, min(J, static_cast<int>((static_cast<long long>(a.budget_ppm) * J + 999999) / 1000000)));
  const int kvh = h / (a.num_q_heads / a.num_kv_heads);
  const int nqb = ri.nqb;
  const int64_t sbase = a.sc_off[b] + static_cast<int64_t>(h) * nqb * nqb + static_cast<int64_t>(i) * nqb;
  const int r0 = i * a.kb, r1 = min((i + 1) * a.kb, ri.R);
  const int64_t rbase = a.row_off[b] + static_cast<int64_t>(h) * ri.R;

  // HRM flags of the candidates (exact, from the float64 row maxima)
  for (int j = tid; j < J; j += blockDim.x) hrm[j] = 0;
  __syncthreads();
  if (tid < 32) {
    for (int r = r0; r < r1; ++r) {
      const int fl = a.rflags[rbase + r];
      if (fl & 2) continue;
      if (fl & 1) {
        const uint32_t* bits = a.hrm_bits + (rbase + r) * a.words_per_row;
        for (int j = tid; j < J; j += 32)
          if ((bits[j >> 5] >> (j & 31)) & 1u) hrm[j] = 1;
      } else if (tid == 0) {
        hrm[(a.c1[rbase + r] * a.stride) / a.block_size] = 1;
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // sort keys (bitonic, descending) over the next power of two
  int n2 = 1;
  while (n2 < J) n2 <<= 1;
  for (int j = tid; j < n2; j += blockDim.x)
    key[j] = (j < J) ? sort_key(hrm[j] != 0, fmaxf(a.score[sbase + j], 0.0f), j) : 0ull;
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int x = tid; x < n2; x += blockDim.x) {
        const int y = x ^ jj;
        if (y > x) {
          const unsigned long long kx = key[x], ky = key[y];
          const bool desc = (x & k) == 0;
          if (desc ? (kx < ky) : (kx > ky)) { key[x] = ky; key[y] = kx; }
        }
      }
      __syncthreads();
    }
  }
  // score intervals per sorted position
  if (tid == 0) {
    n_rep_s = 0;
    int nh = 0;
    while (nh < J && (key[nh] >> 63)) ++nh;
    n_hrm_s = nh;
  }
  for (int p = tid; p < n2; p += blockDim.x) {
    if (p < J) {
      const int j = key_block(key[p]);
      const float s = fmaxf(a.score[sbase + j], 0.0f);
      const float e = a.score_err[sbase + j];
      lo[p] = s - e;
      hi[p] = s + e;
    } else {
      lo[p] = -INFINITY;
      hi[p] = -INFINITY;
    }
  }
  __syncthreads();
  const int nh = n_hrm_s;
  // suffix maximum of hi inside each group (Hillis-Steele, log2(n2) rounds)
  for (int p = tid; p < n2; p += blockDim.x) suf[p] = hi[p];
  __syncthreads();
  for (int off = 1; off < n2; off <<= 1) {
    float tmp[16];
    int cnt = 0;
    for (int p = tid; p < n2; p += blockDim.x, ++cnt) {
      const int q = p + off;
      const bool same = q < n2 && ((p < nh) == (q < nh));
      tmp[cnt & 15] = same ? fmaxf(suf[p], suf[q]) : suf[p];
    }
    __syncthreads();
    cnt = 0;
    for (int p = tid; p < n2; p += blockDim.x, ++cnt) suf[p] = tmp[cnt & 15];
    __syncthreads();
  }
  // clusters of positions whose relative order, or side of the budget cut, the bounds cannot
  // certify: [p, q] grows while some later element of the group may exceed its lowest member
  if (tid == 0) {
    int nr = 0;
    for (int g = 0; g < 2; ++g) {
      const int g0 = g == 0 ? 0 : nh, g1 = g == 0 ? nh : J;
      int p = g0;
      while (p < g1 && p < K) {
        float cmin = lo[p];
        int q = p;
        while (q + 1 < g1 && suf[q + 1] >= cmin) {
          ++q;
          cmin = fminf(cmin, lo[q]);
        }
        if (q > p)
          for (int x = p; x <= q; ++x) rep_pos[nr++] = x;
        p = q + 1;
      }
    }
    n_rep_s = nr;
  }
  __syncthreads();
  const int n_rep = n_rep_s;
  if (n_rep > 0) {
    // exact scores, one warp per repaired block: s_ij = sum over rows r (ascending) of
    // exp(bm[r,j] - M_r) with float64 logits
    const int warps = blockDim.x / 32, w = tid >> 5, lane = tid & 31;
    const float sc = static_cast<float>(a.sm_scale);
    for (int m = w; m < n_rep; m += warps) {
      const int j = key_block(key[rep_pos[m]]);
      double sum = 0.0;
      for (int r = r0; r < r1; ++r) {
        const int64_t rec = rbase + r;
        const double Mr = a.M[rec];
        if (Mr == -INFINITY) continue;
        const uint16_t* qr = query_ptr(a, ri, h, r);
        const float e_r = a.err[rec];
        float mx = -INFINITY;
        for (int c = 0; c < a.kb; ++c) {
          const int kc = j * a.kb + c;
          const uint16_t* kp = (kc <= r) ? key_ptr(a, ri, b, kvh, kc) : nullptr;
          if (kp != nullptr) mx = fmaxf(mx, warp_dot_f32<HD>(qr, kp) * sc);
        }
        if (mx == -INFINITY) continue;
        double bm = -INFINITY;
        for (int c = 0; c < a.kb; ++c) {
          const int kc = j * a.kb + c;
          const uint16_t* kp = (kc <= r) ? key_ptr(a, ri, b, kvh, kc) : nullptr;
          if (kp == nullptr) continue;
          if (warp_dot_f32<HD>(qr, kp) * sc < mx - 2.0f * e_r) continue;
          bm = fmax(bm, warp_dot_f64<HD>(qr, kp) * a.sm_scale);
        }
        sum += exp(bm - Mr);
      }
      if (lane == 0) rep_val[m] = sum;
    }
    __syncthreads();
    // re-sort the repaired runs by (exact score desc, block asc); a run never crosses the
    // HRM / rest boundary
    if (tid == 0) {
      int m0 = 0;
      while (m0 < n_rep) {
        int m1 = m0;
        while (m1 + 1 < n_rep && rep_pos[m1 + 1] == rep_pos[m1] + 1 && rep_pos[m1 + 1] != nh) ++m1;
        for (int x = m0 + 1; x <= m1; ++x) {
          const double vx = rep_val[x];
          const unsigned long long kx = key[rep_pos[x]];
          int y = x - 1;
          while (y >= m0) {
            const double vy = rep_val[y];
            const unsigned long long ky = key[rep_pos[y]];
            const bool before = (vx > vy) || (vx == vy && key_block(kx) < key_block(ky));
            if (!before) break;
            rep_val[y + 1] = vy;
            key[rep_pos[y + 1]] = ky;
            --y;
          }
          rep_val[y + 1] = vx;
          key[rep_pos[y + 1]] = kx;
        }
        m0 = m1 + 1;
      }
    }
    __syncthreads();
  }
  for (int k = tid; k < a.mask_pitch; k += blockDim.x) out[k] = (k < K) ? key_block(key[k]) : -1;
  if (tid == 0) a.mask_len[mrow] = K;
}

template <typename T>
T* carve(uint8_t*& p, size_t n) {
  uintptr_t x = (reinterpret_cast<uintptr_t>(p) + 255) & ~uintptr_t(255);
  T* r = reinterpret_cast<T*>(x);
  p = reinterpret_cast<uint8_t*>(x + n * sizeof(T));
  return r;
}

struct WsLayout {
  size_t rows, scores, words;
};

WsLayout ws_layout(int num_reqs, int num_q_heads, int block_size, int stride, int total_tokens, int max_seqlen) {
  WsLayout w;
  const size_t nqb_max = (max_seqlen + block_size - 1) / block_size;
  w.rows = static_cast<size_t>(num_q_heads) * (static_cast<size_t>(total_tokens) / stride + num_reqs);
  w.scores = static_cast<size_t>(num_q_heads) * nqb_max * (static_cast<size_t>(total_tokens) / block_size + num_reqs);
  w.words = (nqb_max + 31) / 32;
  return w;
}

template <int HD, int KB>
cudaError_t launch_kap_t(KapArgs a, cudaStream_t stream) {
  const int threads = 128;
  kap_setup_kernel<<<1, 256, 0, stream>>>(a);
  {
    dim3 g((a.max_seqlen / a.stride + 1 + 255) / 256, a.num_reqs * a.num_kv_heads);
    kap_knorm_kernel<HD><<<g, 256, 0, stream>>>(a);
  }
  const size_t tsm = sizeof(KapTileSmem<HD>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kap_logits_kernel<HD, KB, kModeRowMax>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(tsm));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kap_logits_kernel<HD, KB, kModeScores>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(tsm));
  if (e != cudaSuccess) return e;
  const unsigned tiles = static_cast<unsigned>(a.num_reqs) * a.num_q_heads * a.nrow_tiles_max;
  kap_logits_kernel<HD, KB, kModeRowMax><<<tiles, threads, tsm, stream>>>(a);
  {
    const size_t rows = static_cast<size_t>(a.num_q_heads) * (static_cast<size_t>(a.total_tokens) / a.stride + a.num_reqs);
    const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
    kap_exact_kernel<HD><<<blocks, 256, 0, stream>>>(a);
  }
  kap_logits_kernel<HD, KB, kModeScores><<<tiles, threads, tsm, stream>>>(a);
  int cap = 32;
  while (cap < a.nqb_max) cap <<= 1;
  const size_t ssm = select_smem_bytes(cap);
  e = cudaFuncSetAttribute(kap_select_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ssm));
  if (e != cudaSuccess) return e;
  kap_select_kernel<HD><<<static_cast<unsigned>(a.num_reqs) * a.num_q_heads * a.nqb_max, kSelectThreads, ssm, stream>>>(a, cap);
  return cudaGetLastError();
}

}  // namespace

size_t kap_workspace_bytes(int num_reqs, int num_q_heads, int num_kv_heads, int block_size, int stride,
                           int total_tokens, int max_seqlen) {
  const WsLayout w = ws_layout(num_reqs, num_q_heads, block_size, stride, total_tokens, max_seqlen);
  size_t n = 0;
  auto add = [&](size_t bytes) { n = ((n + 255) & ~size_t(255)) + bytes; };
  add(sizeof(int64_t) * (num_reqs + 1));
  add(sizeof(int64_t) * (num_reqs + 1));
  add(sizeof(float) * num_reqs * num_kv_heads);
  add(sizeof(float) * static_cast<size_t>(num_reqs) * num_kv_heads * ((max_seqlen + block_size - 1) / block_size));
  add(sizeof(float) * w.rows * kTop);
  add(sizeof(int32_t) * w.rows * kTop);
  add(sizeof(float) * w.rows);
  add(sizeof(int32_t) * w.rows);
  add(sizeof(double) * w.rows);
  add(sizeof(float) * w.rows);
  add(sizeof(int32_t) * w.rows);
  add(sizeof(uint32_t) * w.rows * w.words);
  add(sizeof(float) * w.scores);
  add(sizeof(float) * w.scores);
  return n + 256;
}

cudaError_t kap_static_scratch(void** ptr) {
  // Host code cannot use the array's name as a device address: look the address up, once per
  // device, with that device current.
  static std::mutex mu;
  static void* addr[kMaxStaticDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxStaticDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, cosa_kap_static_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

cudaError_t launch_kap(const KapLaunch& L, cudaStream_t stream) {
  KapArgs a{};
  a.q = L.q;
  a.cu_seqlens = L.cu_seqlens;
  a.k_cache = L.k_cache;
  a.page_table = L.page_table;
  a.mask = L.mask;
  a.mask_len = L.mask_len;
  a.status = L.status;
  a.num_reqs = L.num_reqs;
  a.num_q_heads = L.num_q_heads;
  a.num_kv_heads = L.num_kv_heads;
  a.head_dim = L.head_dim;
  a.block_size = L.block_size;
  a.page_size = L.page_size;
  a.stride = L.stride;
  a.kb = L.block_size / L.stride;
  a.total_tokens = L.total_tokens;
  a.max_seqlen = L.max_seqlen;
  a.num_pages = L.num_pages;
  a.max_pages_per_req = L.max_pages_per_req;
  a.mask_pitch = L.mask_pitch;
  a.budget_ppm = L.budget_ppm;
  a.sm_scale = L.sm_scale;
  a.nqb_max = (L.max_seqlen + L.block_size - 1) / L.block_size;
  const int rmax = (L.max_seqlen + L.stride - 1) / L.stride;
  a.nrow_tiles_max = (rmax + kRowTile - 1) / kRowTile;
  const WsLayout w = ws_layout(L.num_reqs, L.num_q_heads, L.block_size, L.stride, L.total_tokens, L.max_seqlen);
  a.words_per_row = static_cast<int>(w.words);
  uint8_t* p = static_cast<uint8_t*>(L.workspace);
  a.row_off = carve<int64_t>(p, L.num_reqs + 1);
  a.sc_off = carve<int64_t>(p, L.num_reqs + 1);
  a.knorm = carve<float>(p, static_cast<size_t>(L.num_reqs) * L.num_kv_heads);
  a.kbnorm = carve<float>(p, static_cast<size_t>(L.num_reqs) * L.num_kv_heads * a.nqb_max);
  a.topv = carve<float>(p, w.rows * kTop);
  a.topc = carve<int32_t>(p, w.rows * kTop);
  a.qnorm = carve<float>(p, w.rows);
  a.c1 = carve<int32_t>(p, w.rows);
  a.M = carve<double>(p, w.rows);
  a.err = carve<float>(p, w.rows);
  a.rflags = carve<int32_t>(p, w.rows);
  a.hrm_bits = carve<uint32_t>(p, w.rows * w.words);
  a.score = carve<float>(p, w.scores);
  a.score_err = carve<float>(p, w.scores);
  if (static_cast<size_t>(p - static_cast<uint8_t*>(L.workspace)) > L.workspace_bytes) return cudaErrorInvalidValue;
  const int kb = a.kb;
  if (L.head_dim == 128) {
    if (kb == 8) return launch_kap_t<128, 8>(a, stream);
    if (kb == 4) return launch_kap_t<128, 4>(a, stream);
    if (kb == 16) return launch_kap_t<128, 16>(a, stream);
  } else if (L.head_dim == 64) {
    if (kb == 8) return launch_kap_t<64, 8>(a, stream);
    if (kb == 4) return launch_kap_t<64, 4>(a, stream);
    if (kb == 16) return launch_kap_t<64, 16>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace cosa
