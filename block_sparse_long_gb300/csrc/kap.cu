// Kernel-Aware Proxy (KAP): computation-order mask from stride-sampled queries and keys.
//
// CoSA (arXiv 2607.25291) Sec. 4.2, Eqs. (8)-(14), Algorithm A (proxy stage).  For each
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
// get wrong is settled at float64 accuracy or better.  The kernels, in launch order:
//   kap_setup                per-request offsets into the workspace, zeroed key norms;
//   kap_gather               the sampled queries and keys packed into contiguous 128-row padded
//                            arrays, a validity bit per key, the largest key norm per key block;
//   kap_logits               one tensor-core pass over every causal (sampled row, sampled key) tile:
//                            per row the largest fp32 logit, its key and the largest over the other
//                            keys, and per (row, key block) the block maximum of Eq. (9), stored;
//   kap_exact                per row: error bound e_r >= |fp32 logit - exact logit| for every key of
//                            the row (from ||q_r|| * max ||k|| and the accumulation model of kKappa);
//                            if the runner-up is more than 2 e_r below the maximum the argmax key is
//                            certain and M_r is its exact logit (three-term fp32 sum);
//   kap_rescan               rows where it is not: every key of the blocks whose stored fp32 block
//                            maximum is within 3 e_r of the largest logit is re-evaluated in float64;
//                            the HRM blocks of the row follow exactly;
//   kap_block_scores         per (query block, key block): fp32 score from the stored block maxima
//                            and the exact M_r, with a rigorous bound on its error;
//   kap_select_warp          a warp per mask row: top-K by radix select, sort, certification of
//                            every adjacent pair and of the budget cut against the bounds, float64
//                            repair of the uncertain positions; rows it cannot settle are listed;
//   kap_select               a block per listed row: the same with a full sort (top-p, ascending
//                            order, long rows, cuts the sentinel cannot certify).
#include <cstdint>
#include <mutex>
#include <type_traits>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "cosa.h"
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
  float* v1;             // per sampled row: largest fp32 logit (scaled), -inf if none
  float* v2;             // per sampled row: largest fp32 logit over the other keys (scaled)
  int32_t* c1;           // per sampled row: key of v1, then the exact argmax key (first if several tie)
  int64_t* amb;          // [0] = count, [1..] = rows whose maximum is not certain from fp32

  float* qnorm;          // per sampled row: ||q~_r|| rounded up
  double* M;             // per sampled row: exact maximum logit (scaled), -inf if none
  float* err;            // per sampled row: error bound e_r of its fp32 logits (scaled)
  int32_t* rflags;       // per sampled row: bit 0 = several HRM candidates (bitmap valid), bit 1 = empty
  uint32_t* hrm_bits;    // per sampled row: bitmap of HRM blocks, words_per_row words (ambiguous rows only)
  float* score;          // per (request, head): nqb x nqb fp32 scores, row i = query block
  float* score_err;      // same shape: bound on |score - exact score|
  int64_t* qs_off;       // [B+1]: first gathered query row of request b (times Hq), rows padded to 128
  int64_t* ks_off;       // [B+1]: first gathered key row of request b (times Hkv), rows padded to 128
  uint16_t* qs;          // gathered sampled queries, bf16 [rows, d]: row qs_off[b] + h * Rp + r
  uint16_t* ks;          // gathered sampled keys, bf16 [rows, d]: row ks_off[b] + kvh * Rp + c (zero if absent)
  uint32_t* kvalid;      // one bit per gathered key row: the key exists
  int32_t* defer;        // [0] = count, [1..] = mask rows left to the block-per-row select kernel
  int64_t* bm_off;       // [B+1]: first block maximum of request b (times Hq)
  float* bm;             // per (request, head, sampled row r, key block j <= r / kb): the largest
                         // visible fp32 logit of block j (raw, unscaled), -inf if none
  int num_reqs, num_q_heads, num_kv_heads, head_dim, block_size, page_size, stride, kb;
  int total_tokens, max_seqlen, num_pages, max_pages_per_req, mask_pitch, budget_ppm;
  int nqb_max, nrow_tiles_max, words_per_row;
  double sm_scale;
  int ascending;         // write the selected blocks in ascending block order
  int top_p;             // budget_ppm is the top-p threshold p, not the fraction B1
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

// Block maxima layout: per (request, head), query block i holds (i + 1) rounded up to 64 / kb key
// blocks (its pitch), each as the kb maxima of its sampled rows in row order: the maximum of key
// block j for row q of the query block is element j * kb + q.  The kb lanes of the logits epilogue
// that hold a query block's rows then store each key block's maxima as kb consecutive floats, and
// the block-score kernel reads them as one vector per key block.
// floats before query block i (sum over i' < i of kb times the pitch of i')
__host__ __device__ __forceinline__ int64_t bm_block_base(int i, int kb) {
  const int64_t ng = 64 / kb;
  const int64_t full = i / ng;                   // complete groups of ng query blocks
  // blocks g*ng .. g*ng + ng - 1 have pitch (g + 1) * ng
  int64_t sum = ng * ng * full * (full + 1) / 2 + (i - full * ng) * (full + 1) * ng;
  return kb * sum;
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

// eight bf16 values from a 16-byte aligned address, widened to fp32
// per-thread asynchronous copies into shared memory (16 bytes each, both addresses 16-byte aligned),
// completing in commit groups
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most N of this thread's commit groups are still in flight
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void load8_bf16(const uint16_t* p, float (&f)[8]) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// ---------------------------------------------------------------------------
// setup: per-request offsets into the workspace, zeroed key norms, input checks
// ---------------------------------------------------------------------------
__global__ void kap_setup_kernel(KapArgs a) {
  if (threadIdx.x == 0) {
    int64_t ro = 0, so = 0, qo = 0, ko = 0, bo = 0;
    for (int b = 0; b < a.num_reqs; ++b) {
      a.row_off[b] = ro;
      a.sc_off[b] = so;
      a.qs_off[b] = qo;
      a.ks_off[b] = ko;
      a.bm_off[b] = bo;
      const ReqInfo ri = req_info(a, b);
      if (!ri.ok) report_status(a.status, kStatusBadInput);
      const int64_t rp = (ri.R + kRowTile - 1) / kRowTile * kRowTile;
      ro += static_cast<int64_t>(a.num_q_heads) * ri.R;
      so += static_cast<int64_t>(a.num_q_heads) * ri.nqb * ri.nqb;
      qo += static_cast<int64_t>(a.num_q_heads) * rp;
      ko += static_cast<int64_t>(a.num_kv_heads) * rp;
      bo += static_cast<int64_t>(a.num_q_heads) * bm_block_base(ri.nqb, a.kb);
    }
    a.bm_off[a.num_reqs] = bo;
    a.row_off[a.num_reqs] = ro;
    a.sc_off[a.num_reqs] = so;
    a.qs_off[a.num_reqs] = qo;
    a.ks_off[a.num_reqs] = ko;
    a.amb[0] = 0;
    a.defer[0] = 0;
  }
  for (int e = threadIdx.x; e < a.num_reqs * a.num_kv_heads; e += blockDim.x) a.knorm[e] = 0.0f;
  for (int e = threadIdx.x; e < a.num_reqs * a.num_kv_heads * a.nqb_max; e += blockDim.x) a.kbnorm[e] = 0.0f;
}

// Gather the stride-sampled queries and keys of every (request, head) into contiguous, 128-row
// padded arrays (absent keys and padding rows are zero), record which keys exist, and the largest
// key norm per (request, kv head) and per key block.  One warp per 32 rows, eight rows in flight;
// each lane moves HD / 32 consecutive elements of a row with one vector load and store.  grid.y
// walks the requests' q heads then kv heads.
template <int HD>
__global__ void __launch_bounds__(256) kap_gather_kernel(KapArgs a) {
  constexpr int PER = HD / 32;  // bf16 per lane per row
  static_assert(PER == 4 || PER == 2, "d = 128 or 64");
  using Vec = typename std::conditional<PER == 4, uint2, uint32_t>::type;
  const int nh = a.num_q_heads + a.num_kv_heads;
  const int b = blockIdx.y / nh, hh = blockIdx.y % nh;
  const bool is_key = hh >= a.num_q_heads;
  const ReqInfo ri = req_info(a, b);
  const int rp = (ri.R + kRowTile - 1) / kRowTile * kRowTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = (blockIdx.x * 8 + warp) * 32;
  if (r0 >= rp) return;
  const int head = is_key ? hh - a.num_q_heads : hh;
  const int64_t base = is_key ? a.ks_off[b] + static_cast<int64_t>(head) * rp : a.qs_off[b] + static_cast<int64_t>(head) * rp;
  uint16_t* dst_base = (is_key ? a.ks : a.qs) + base * HD;
  constexpr int U = 8;          // rows in flight
  uint32_t valid_bits = 0;
  float blk_norm = 0.0f;        // running max over the rows of the current key block
  for (int rr0 = 0; rr0 < 32; rr0 += U) {
    Vec val[U];
    bool have[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = r0 + rr0 + u;
      const uint16_t* src = nullptr;
      if (r < ri.R) src = is_key ? key_ptr(a, ri, b, head, r) : query_ptr(a, ri, head, r);
      have[u] = src != nullptr;
      if (src) val[u] = *reinterpret_cast<const Vec*>(src + lane * PER);
      else val[u] = Vec{};
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int rr = rr0 + u;
      const int r = r0 + rr;
      *reinterpret_cast<Vec*>(dst_base + static_cast<int64_t>(r) * HD + lane * PER) = val[u];
      if (is_key) {
        uint32_t w[2];
        if constexpr (PER == 4) {
          w[0] = val[u].x;
          w[1] = val[u].y;
        } else {
          w[0] = val[u];
          w[1] = 0u;
        }
        float s2 = 0.0f;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
          const float x = __uint_as_float((e & 1) ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16));
          s2 = fmaf(x, x, s2);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        const float nrm = have[u] ? sqrtf(s2) * (1.0f + 1.0f / 65536.0f) : 0.0f;
        if (have[u]) valid_bits |= 1u << rr;
        blk_norm = fmaxf(blk_norm, nrm);
        const int j = (r * a.stride) / a.block_size;
        const bool last_of_block = (rr == 31) || (((r + 1) * a.stride) / a.block_size != j);
        if (last_of_block && lane == 0 && blk_norm > 0.0f) {
          atomicMax(reinterpret_cast<int*>(&a.kbnorm[(static_cast<size_t>(b) * a.num_kv_heads + head) * a.nqb_max + j]),
                    __float_as_int(blk_norm));
          atomicMax(reinterpret_cast<int*>(&a.knorm[b * a.num_kv_heads + head]), __float_as_int(blk_norm));
        }
        if (last_of_block) blk_norm = 0.0f;
      }
    }
  }
  if (is_key && lane == 0) a.kvalid[(base + r0) >> 5] = valid_bits;
}

// ---------------------------------------------------------------------------
// sampled logits on tcgen05: 128 sampled rows x all causal sampled keys
// ---------------------------------------------------------------------------
constexpr int kKeyStages = 2;           // K~ tiles in flight (two CTAs fit per SM)
constexpr int kMaxKeyTiles = 512;       // key tiles of the longest request: 4096 query blocks of 16 sampled rows
constexpr int kLogitsThreads = 320;      // warp 0 TMA, warp 1 UMMA, warps 2-9 epilogue

template <int HD>
struct alignas(1024) KapTileSmem {
  uint8_t q[kRowTile * HD * 2];          // [HD/64][128][128 B] SW128
  uint8_t k[kKeyStages][kKeyTile * HD * 2];
  uint64_t q_full;
  uint64_t k_full[kKeyStages], k_free[kKeyStages];
  uint64_t acc_full[2], acc_free[2];
  uint64_t cleanup;
  float hv1[2][128], hv2[2][128];        // per column half: the row's largest and second largest logit
  int32_t hc1[2][128];
  uint32_t kval[kMaxKeyTiles * 4];       // validity bits of the row tile's causal keys (4 words per key tile)
  uint32_t tmem_base;
  int32_t abort_flag;
};

// Sampled logits l = q~ . k~ (fp32, tcgen05) for 128 sampled rows against every causal key tile of
// 128 sampled keys.  The epilogue keeps the two largest logits of each row and the key of the first
// (candidates for the exact maximum) and stores, per (row, key block j <= the row's query block), the
// block maximum of Eq. (9) before normalisation; kap_block_scores_kernel turns those into s_ij once
// the float64 row maxima are known.
// Warp 0 streams the K~ tiles with TMA, warp 1 issues the UMMAs into two TMEM accumulators, warps
// 2-9 read the accumulators: warp w serves TMEM lanes 32 (w % 4) .. + 31 and columns [64 g, 64 g + 64)
// with g = (w - 2) / 4.
template <int HD, int KB>
__global__ void __launch_bounds__(kLogitsThreads, 2)
    kap_logits_kernel(const __grid_constant__ CUtensorMap qs_map, const __grid_constant__ CUtensorMap ks_map,
                      KapArgs a) {
  using S = KapTileSmem<HD>;
  constexpr int DH = HD / 64;
  constexpr int TILE = kKeyTile * HD * 2;
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
  const int rp = (ri.R + kRowTile - 1) / kRowTile * kRowTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkt = rt + 1;                       // causal key tiles
  const int64_t qrow0 = a.qs_off[b] + static_cast<int64_t>(h) * rp + static_cast<int64_t>(rt) * kRowTile;
  const int64_t krow0 = a.ks_off[b] + static_cast<int64_t>(kvh) * rp;
  volatile int* abort_flag = &sm.abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    for (int st = 0; st < kKeyStages; ++st) { mbar_init(&sm.k_full[st], 1); mbar_init(&sm.k_free[st], 1); }
    for (int st = 0; st < 2; ++st) { mbar_init(&sm.acc_full[st], 1); mbar_init(&sm.acc_free[st], 8); }
    mbar_init(&sm.cleanup, 1);
    sm.abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    int issued = 0;
    if (lane == 0) {
      tma_prefetch_desc(&qs_map);
      tma_prefetch_desc(&ks_map);
      mbar_arrive_expect_tx(&sm.q_full, kRowTile * HD * 2);
      for (int dh = 0; dh < DH; ++dh)
        tma_load_2d(&sm.q[dh * 128 * 128], &qs_map, &sm.q_full, dh * 64, static_cast<int>(qrow0));
      for (int kt = 0; kt < nkt; ++kt) {
        const int st = kt % kKeyStages;
        if (kt >= kKeyStages && !wait_parity_bounded(&sm.k_free[st], ((kt / kKeyStages) - 1) & 1, abort_flag, a.status))
          break;
        mbar_arrive_expect_tx(&sm.k_full[st], TILE);
        for (int dh = 0; dh < DH; ++dh)
          tma_load_2d(&sm.k[st][dh * 128 * 128], &ks_map, &sm.k_full[st], dh * 64,
                      static_cast<int>(krow0 + static_cast<int64_t>(kt) * kKeyTile));
        ++issued;
      }
      if (*abort_flag) {
        wait_parity_bounded(&sm.q_full, 0, nullptr, nullptr);
        for (int st = 0; st < kKeyStages; ++st) {
          const int n = (issued - st + kKeyStages - 1) / kKeyStages;
          if (n > 0) wait_parity_bounded(&sm.k_full[st], (n - 1) & 1, nullptr, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ UMMA issuer ------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kKeyTile, false, false);
      bool ok = wait_parity_bounded(&sm.q_full, 0, abort_flag, a.status);
      tc_fence_after();
      for (int kt = 0; ok && kt < nkt; ++kt) {
        const int st = kt % kKeyStages, ab = kt & 1;
        if (!wait_parity_bounded(&sm.k_full[st], (kt / kKeyStages) & 1, abort_flag, a.status)) break;
        if (kt >= 2 && !wait_parity_bounded(&sm.acc_free[ab], ((kt >> 1) - 1) & 1, abort_flag, a.status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint64_t ad = smem_desc_sw128(smem_u32(&sm.q[(kk >> 2) * 128 * 128 + (kk & 3) * 32]), 16, 1024);
          const uint64_t bd = smem_desc_sw128(smem_u32(&sm.k[st][(kk >> 2) * 128 * 128 + (kk & 3) * 32]), 16, 1024);
          umma_ss(tmem + ab * 128, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(&sm.acc_full[ab]);
        umma_commit(&sm.k_free[st]);
      }
      umma_commit(&sm.cleanup);
      wait_parity_bounded(&sm.cleanup, 0, nullptr, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------ epilogue (warps 2-9) ------------------------------
    const int g = (warp - 2) >> 2;                // column half
    const int t = (warp & 3) * 32 + lane;         // row in the tile == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int r = rt * kRowTile + t;              // sampled row
    const bool row_ok = r < ri.R;
    const int64_t rec = a.row_off[b] + static_cast<int64_t>(h) * ri.R + r;
    const float scale = static_cast<float>(a.sm_scale);
    const uint32_t* kval = a.kvalid + (krow0 >> 5);
    float r1 = -INFINITY, r2 = -INFINITY;     // largest and second largest raw logit of this half
    int rc1 = -1;
    const int nqb = ri.nqb;
    const int qblk = r / KB;
    // this row's block maxima: element j * KB + (r - qblk * KB) of its query block's region
    float* bm_row = a.bm + a.bm_off[b] + static_cast<int64_t>(h) * bm_block_base(nqb, KB) + bm_block_base(qblk, KB) +
                    (r - qblk * KB);
    // the validity words of every causal key tile, staged once: their loads stay off the per-tile path
    for (int e = threadIdx.x - 64; e < nkt * 4; e += 256) sm.kval[e] = __ldg(kval + e);
    named_bar_sync(2, 256);
    for (int kt = 0; kt < nkt; ++kt) {
      const int ab = kt & 1;
      const uint32_t bits0 = sm.kval[kt * 4 + g * 2], bits1 = sm.kval[kt * 4 + g * 2 + 1];
      const bool okw = __all_sync(0xffffffffu,
                                  wait_parity_bounded(&sm.acc_full[ab], (kt >> 1) & 1, abort_flag, a.status));
      if (!okw) break;
      tc_fence_after();
      // this thread's 64 logits as NG groups of KB columns (one key block each); each load also
      // returns its group's maximum, which is the block maximum when every column is visible
      constexpr int NG = 64 / KB;                 // key blocks in this thread's 64 columns
      uint32_t vv[64];
      float bmh[NG];
#pragma unroll
      for (int gg = 0; gg < NG; ++gg) tmem_ldn_max<KB>(tmem + lane_addr + ab * 128 + g * 64 + gg * KB, &vv[gg * KB], bmh[gg]);
      tmem_wait_ld();
#pragma unroll
      for (int gg = 0; gg < NG; ++gg) reg_after_wait(bmh[gg]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_free[ab]);
      const int c0 = kt * kKeyTile + g * 64;      // key index of this thread's first column
      const int last = r - c0;                    // causal: columns <= last
      // every column of this thread's half is visible: below the diagonal tile, all keys valid
      const bool interior = row_ok && kt < rt && (bits0 & bits1) == 0xffffffffu;
      float bmg[NG];
      if (interior) {
#pragma unroll
        for (int gg = 0; gg < NG; ++gg) bmg[gg] = bmh[gg];
        // tile maximum from the block maxima; the first index and the tile's second largest value
        // are only needed when the running maximum rises (a few tiles per row)
        float t1 = bmg[0];
#pragma unroll
        for (int gg = 1; gg < NG; ++gg) t1 = fmaxf(t1, bmg[gg]);
        if (t1 > r1) {
          int e1 = 0;
#pragma unroll
          for (int e = 63; e >= 0; --e)
            if (__uint_as_float(vv[e]) == t1) e1 = e;
          float t2 = -INFINITY;
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e != e1) t2 = fmaxf(t2, __uint_as_float(vv[e]));
          r2 = fmaxf(r1, t2);
          r1 = t1;
          rc1 = c0 + e1;
        } else {
          r2 = fmaxf(r2, t1);
        }
      } else {
#pragma unroll
        for (int gg = 0; gg < NG; ++gg) bmg[gg] = -INFINITY;
        // branch-free: second max = max(second, min(x, max)); argmax follows the first strict increase
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const uint32_t bits = e < 32 ? bits0 : bits1;
          const bool vis = row_ok && e <= last && ((bits >> (e & 31)) & 1u);
          const float x = vis ? __uint_as_float(vv[e]) : -INFINITY;
          bmg[e / KB] = fmaxf(bmg[e / KB], x);
          r2 = fmaxf(r2, fminf(x, r1));
          rc1 = (x > r1) ? c0 + e : rc1;
          r1 = fmaxf(r1, x);
        }
      }
      // the group of NG blocks starts at a multiple of NG <= qblk, so it fits the padded region; the
      // KB lanes of a query block write KB consecutive floats per key block (whole 32-byte sectors)
      if (row_ok && c0 / KB <= qblk) {
#pragma unroll
        for (int gg = 0; gg < NG; ++gg) bm_row[static_cast<int64_t>(c0 / KB + gg) * KB] = bmg[gg];
      }
    }
    // merge the two column halves; half 0 writes the row's record
    sm.hv1[g][t] = r1;
    sm.hv2[g][t] = r2;
    sm.hc1[g][t] = rc1;
    named_bar_sync(1, 256);
    if (g == 0 && row_ok) {
      const float a1 = sm.hv1[0][t], b1 = sm.hv1[1][t];
      const int ac = sm.hc1[0][t], bc = sm.hc1[1][t];
      const float m1 = fmaxf(a1, b1);
      const float m2 = fmaxf(fminf(a1, b1), fmaxf(sm.hv2[0][t], sm.hv2[1][t]));
      const int mc = (a1 > b1 || (a1 == b1 && ac >= 0)) ? ac : bc;
      a.v1[rec] = (m1 == -INFINITY) ? -INFINITY : m1 * scale;
      a.v2[rec] = (m2 == -INFINITY) ? -INFINITY : m2 * scale;
      a.c1[rec] = mc;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------------------
// block scores (Eqs. (9)-(11)): s_ij = sum over the sampled rows r of query block i of
// Pbar[r, j] = exp(bm[r, j] * scale - M_r), with the float64 row maxima M_r, and a bound on
// |s_ij - exact|.  A block per (request, head, query block), a thread per key block j <= i.
//
// Each term is taken in base 2: x = 2^u, u = bm * (scale log2 e) - M_r log2 e, by the hardware
// exponential, whose relative error is at most kEx2Rel (a test measures it over every input).  The
// first factor is rounded once to fp32; the second three times (M_r to fp32, the fp32 log2 e, their
// product); the fmaf once.  With |bm * scale log2 e| <= |u| + |M_r log2 e| and U the exact exponent,
//   |u - U| <= log2 e * dl * ||k||max_j + 2^-23 |u| + 2^-22 |M_r log2 e|,
// dl = kKappa * scale * ||q_r|| the logit error per unit key norm; and |2^D - 1| <= 1.02 ln 2 |D|
// for |D| <= 0.04.  Hence
//   |x - 2^U| <= x (1 + 2^-19) (kEx2Rel + 1.02 dl ||k||max_j + 1.7e-7 |M_r log2 e| + 8.5e-8 |u|),
// plus 2^-125 for a result the instruction flushes to zero (u < -126: the exact value is below
// 2^-125 too).  Blocks outside that expansion's range take a looser bound through expm1f.
// ---------------------------------------------------------------------------
constexpr float kEx2Rel = 8.0f / 16777216.0f;   // 2^-21: the relative error assumed of ex2.approx.ftz.f32

constexpr int kScoreDepth = 3;   // key blocks in flight per thread in the block-score kernel

template <int KB>
__global__ void __launch_bounds__(128, 8) kap_block_scores_kernel(KapArgs a) {
  const int i = a.nqb_max - 1 - static_cast<int>(blockIdx.x);   // heaviest query blocks first
  const int h = blockIdx.y, b = blockIdx.z;
  const ReqInfo ri = req_info(a, b);
  if (i >= ri.nqb) return;
  const int nqb = ri.nqb;
  const int kvh = h / (a.num_q_heads / a.num_kv_heads);
  const float scale = static_cast<float>(a.sm_scale);
  const float sl2 = static_cast<float>(a.sm_scale * 1.4426950408889634);
  const int64_t rbase = a.row_off[b] + static_cast<int64_t>(h) * ri.R;
  const float* bm_blk = a.bm + a.bm_off[b] + static_cast<int64_t>(h) * bm_block_base(nqb, KB) + bm_block_base(i, KB);
  const float* kbn = a.kbnorm + (static_cast<size_t>(b) * a.num_kv_heads + kvh) * a.nqb_max;
  const int64_t sbase = a.sc_off[b] + static_cast<int64_t>(h) * nqb * nqb + static_cast<int64_t>(i) * nqb;
  constexpr float kGrow = 1.0f + 1.0f / 524288.0f;   // 1 + 2^-19
  constexpr float kRnd = 8.5e-8f;                    // >= 1.02 ln 2 2^-23 (|u|)
  constexpr float kRndM = 1.7e-7f;                   // >= 1.02 ln 2 2^-22 (|M_r log2 e|)
  // a key block's KB row maxima (KB / 4 16-byte vectors) are copied into this thread's slot of a
  // kScoreDepth-stage ring in shared memory by asynchronous copies, kScoreDepth key blocks ahead of
  // the one scored: the bytes in flight do not take registers, and no other thread reads the slot
  __shared__ __align__(16) float s_ring[kScoreDepth][128 * KB];
  auto issue = [&](int j, int st) {
    const float* src = bm_blk + static_cast<int64_t>(j) * KB;
#pragma unroll
    for (int q = 0; q < KB; q += 4) cp_async16(&s_ring[st][threadIdx.x * KB + q], src + q);
  };
#pragma unroll
  for (int k = 0; k < kScoreDepth; ++k) {
    const int j = static_cast<int>(threadIdx.x) + k * static_cast<int>(blockDim.x);
    if (j <= i) issue(j, k);
    cp_async_commit();   // one group per stage, empty past the row
  }
  // per sampled row of the query block, computed once per block (float64 is slow here): M_r log2 e
  // and the bound's parts.  A row without a visible key (M_r = -inf) gets +inf, which makes every u
  // -inf and its terms 0.
  __shared__ float s_ml2[KB], s_a[KB], s_b[KB], s_dl[KB];
  if (threadIdx.x < KB) {
    const int q = threadIdx.x, r = i * KB + q;
    float ml2 = INFINITY, av = 0.0f, bv = 0.0f, dl = 0.0f;
    if (r < ri.R) {
      const float M = static_cast<float>(a.M[rbase + r]);
      if (M != -INFINITY) {
        ml2 = M * 1.44269504f;
        dl = kKappa * scale * a.qnorm[rbase + r] * 1.001f;
        av = kGrow * (kEx2Rel + kRndM * fabsf(ml2));
        bv = kGrow * 1.02f * dl;
      }
    }
    s_ml2[q] = ml2;
    s_a[q] = av;
    s_b[q] = bv;
    s_dl[q] = dl;
  }
  __syncthreads();
  float Ml2[KB], A[KB], B[KB];
  float dl_max = 0.0f, ml_max = 0.0f;
#pragma unroll
  for (int q = 0; q < KB; ++q) {
    Ml2[q] = s_ml2[q];
    A[q] = s_a[q];
    B[q] = s_b[q];
    dl_max = fmaxf(dl_max, s_dl[q]);
    if (A[q] != 0.0f) ml_max = fmaxf(ml_max, fabsf(Ml2[q]));
  }
  const float C = kGrow * kRnd;
  const bool tail_rows = (i + 1) * KB > ri.R;
  int st = 0;
  for (int j = threadIdx.x; j <= i; j += blockDim.x) {
    const float kbv = __ldg(kbn + j);
    cp_async_wait<kScoreDepth - 1>();   // this key block's group is complete
    float bmv[KB];
#pragma unroll
    for (int q = 0; q < KB; q += 4) {
      const float4 v4 = *reinterpret_cast<const float4*>(&s_ring[st][threadIdx.x * KB + q]);
      bmv[q] = v4.x;
      bmv[q + 1] = v4.y;
      bmv[q + 2] = v4.z;
      bmv[q + 3] = v4.w;
    }
    // rows past the request's sampled rows hold nothing (only a request's last query block has any)
    if (tail_rows) {
#pragma unroll
      for (int q = 0; q < KB; ++q)
        if (i * KB + q >= ri.R) bmv[q] = -INFINITY;
    }
    float x[KB];
    float xe = 0.0f;
    if (dl_max * kbv <= 0.013f && ml_max <= 1.0e5f) {
#pragma unroll
      for (int q = 0; q < KB; ++q) {
        const float u = fmaf(bmv[q], sl2, -Ml2[q]);
        x[q] = ex2_approx(u);
        const float t = fmaf(C, fminf(fabsf(u), 1024.0f), fmaf(B[q], kbv, A[q]));
        xe = fmaf(x[q], t, xe);
      }
    } else {
      // far outside the usual range: D may exceed 0.04, take |2^D - 1| <= expm1(ln 2 |D|) directly
#pragma unroll
      for (int q = 0; q < KB; ++q) {
        x[q] = 0.0f;
        if (A[q] == 0.0f) continue;   // a row without a visible key
        const float u = fmaf(bmv[q], sl2, -Ml2[q]);
        x[q] = ex2_approx(u);
        const float D = 1.4426950408889634f * B[q] / (kGrow * 1.02f) * kbv +
                        1.2e-7f * (2.0f * fabsf(Ml2[q]) + fminf(fabsf(u), 1.0e30f));
        const float rel = expm1f(0.6931472f * D) * 1.01f + kEx2Rel * 1.01f;
        xe = fmaf(x[q], kGrow * rel, xe);
      }
    }
    // pairwise sum over the rows (log2 KB levels)
#pragma unroll
    for (int o = KB / 2; o > 0; o >>= 1) {
#pragma unroll
      for (int q = 0; q < o; ++q) x[q] += x[q + o];
    }
    a.score[sbase + j] = x[0];
    // the fmaf chain's own roundings, the pairwise sum's, and the flushed results
    a.score_err[sbase + j] = xe * kGrow + x[0] * (4.0f * 6.0e-8f) + KB * 2.36e-38f;
    // refill the slot kScoreDepth key blocks ahead: issued after the stores above, which wait for
    // the slot's values, so the copy cannot overtake their reads
    const int jn = j + kScoreDepth * static_cast<int>(blockDim.x);
    if (jn <= i) issue(jn, st);
    cp_async_commit();
    st = (st + 1 == kScoreDepth) ? 0 : st + 1;
  }
}

// ---------------------------------------------------------------------------
// exact row maxima of the sampled rows whose fp32 arg max is certain (kept as float64); four rows
// per warp
// ---------------------------------------------------------------------------
// Sums carried as three fp32 values hi + lo + c.  Knuth's two-sum is an error-free transformation
// (s + e == a + b exactly); every addition is taken through two-sums into the pair (hi, lo) except
// the small third term c, which gathers the pair's own rounding errors.  On sums of 128 bf16
// products this is at least as accurate as a float64 running sum (checked against exact rational
// sums, down to mixed magnitudes 2^-12 .. 2^12), on the FP32 pipe.  The intrinsics keep the
// compiler from contracting or reordering the additions.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
// (hi, lo, c) += y
__device__ __forceinline__ void sum3_add(float& hi, float& lo, float& c, float y) {
  float s, e, t, et;
  two_sum(hi, y, s, e);
  two_sum(e, lo, t, et);
  two_sum(s, t, hi, lo);
  c = __fadd_rn(c, et);
}
// (hi, lo, c) += (yh, yl, yc)
__device__ __forceinline__ void sum3_add(float& hi, float& lo, float& c, float yh, float yl, float yc) {
  float s, e, t, et, t2, et2;
  two_sum(hi, yh, s, e);
  two_sum(e, lo, t, et);
  two_sum(t, yl, t2, et2);
  two_sum(s, t2, hi, lo);
  c = __fadd_rn(__fadd_rn(c, yc), __fadd_rn(et, et2));
}

template <int HD>
__global__ void __launch_bounds__(256) kap_exact_kernel(KapArgs a) {
  // four rows per warp, eight lanes per row: the row's dot product takes three shuffle rounds
  constexpr int RPW = 4, LPR = 32 / RPW, PER = HD / LPR;
  const int lane = threadIdx.x & 31, sub = lane % LPR, grp = lane / LPR;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5)) * RPW + grp;
  const int64_t total = a.row_off[a.num_reqs];
  const bool live = gw < total;
  // locate (b, h, r) of record gw (a lane group past the end works on record 0 and writes nothing)
  const int64_t rec = live ? gw : 0;
  int b = 0;
  while (b + 1 < a.num_reqs && a.row_off[b + 1] <= rec) ++b;
  const ReqInfo ri = req_info(a, b);
  const int64_t local = rec - a.row_off[b];
  const int h = static_cast<int>(local / ri.R);
  const int r = static_cast<int>(local % ri.R);
  const int kvh = h / (a.num_q_heads / a.num_kv_heads);
  const uint16_t* qr = query_ptr(a, ri, h, r) + sub * PER;
  float qf[PER];
#pragma unroll
  for (int e = 0; e < PER; e += 8) {
    float f[8];
    load8_bf16(qr + e, f);
#pragma unroll
    for (int q = 0; q < 8; ++q) qf[e + q] = f[q];
  }
  // ||q_r||
  float s2 = 0.0f;
#pragma unroll
  for (int e = 0; e < PER; ++e) s2 = fmaf(qf[e], qf[e], s2);
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
  const float qn = sqrtf(s2) * (1.0f + 1.0f / 65536.0f);
  // bound on |fp32 logit - exact| for every key of the row (largest key norm of the request)
  const float e_r = kKappa * static_cast<float>(a.sm_scale) * qn * a.knorm[b * a.num_kv_heads + kvh] * 1.001f + 1e-30f;
  const float v1 = a.v1[rec], v2 = a.v2[rec];
  // a key can hold the exact maximum only if its fp32 logit is within 2 e_r of the largest one
  const bool empty = v1 == -INFINITY;
  const bool certain = !empty && v2 < v1 - 2.0f * e_r;
  const uint16_t* kr = certain ? key_ptr(a, ri, b, kvh, a.c1[rec]) + sub * PER : qr;
  // products of two bf16 values are exact in fp32 (8-bit significands); their sum is kept as three
  // fp32 terms on the FP32 pipe (GB300's FP64 pipe runs at a small fraction of that rate and had set
  // this kernel's time when the sum was a float64)
  float hi = 0.0f, lo = 0.0f, cc = 0.0f;
#pragma unroll
  for (int e = 0; e < PER; e += 8) {
    float kf[8];
    load8_bf16(kr + e, kf);
#pragma unroll
    for (int q = 0; q < 8; ++q) sum3_add(hi, lo, cc, __fmul_rn(qf[e + q], kf[q]));
  }
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, hi, o), ol = __shfl_xor_sync(0xffffffffu, lo, o);
    const float oc = __shfl_xor_sync(0xffffffffu, cc, o);
    sum3_add(hi, lo, cc, oh, ol, oc);
  }
  const double acc = (static_cast<double>(hi) + static_cast<double>(lo)) + static_cast<double>(cc);
  if (!live || sub != 0) return;
  a.qnorm[rec] = qn;
  a.err[rec] = e_r;
  if (empty) {
    a.M[rec] = -INFINITY;
    a.rflags[rec] = 2;
    a.c1[rec] = -1;
  } else if (certain) {
    a.M[rec] = acc * a.sm_scale;
    a.rflags[rec] = 0;
  } else {
    // not certain from fp32: settled by kap_rescan_kernel
    a.rflags[rec] = 1;
    const unsigned long long slot = atomicAdd(reinterpret_cast<unsigned long long*>(&a.amb[0]), 1ull);
    a.amb[1 + slot] = rec;
  }
}

// q . k over d = 32 * PER elements, the warp's lanes holding PER each, summed as three fp32 terms
// (bf16 products are exact in fp32) and returned in float64 to every lane (lane 0's sum).
template <int PER>
__device__ __forceinline__ double warp_dot3(const float (&qf)[PER], const float (&kf)[PER]) {
  float hi = 0.0f, lo = 0.0f, cc = 0.0f;
#pragma unroll
  for (int e = 0; e < PER; ++e) sum3_add(hi, lo, cc, __fmul_rn(qf[e], kf[e]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, hi, o), ol = __shfl_xor_sync(0xffffffffu, lo, o);
    const float oc = __shfl_xor_sync(0xffffffffu, cc, o);
    sum3_add(hi, lo, cc, oh, ol, oc);
  }
  const double v = (static_cast<double>(hi) + static_cast<double>(lo)) + static_cast<double>(cc);
  return __shfl_sync(0xffffffffu, v, 0);
}

// Rows whose maximum fp32 cannot certify: a warp per row (warp-stride over the queue).  A key can
// hold the exact maximum only if its fp32 logit is at least v1 - 2 e_r (its exact logit is within
// e_r of its fp32 one, and the exact maximum is at least the fp32 argmax's exact logit, v1 - e_r),
// so only the key blocks whose stored fp32 block maximum (the logits pass) reaches v1 - 3 e_r are
// examined: every visible key of those blocks is evaluated in float64 (lanes split d, butterfly sum:
// every lane holds the same value), the row maximum is the largest, and the row's HRM bitmap flags
// the blocks of the keys that attain it.
template <int HD, int KB>
__global__ void __launch_bounds__(256) kap_rescan_kernel(KapArgs a) {
  constexpr int PER = HD / 32;   // d elements per lane
  const int lane = threadIdx.x & 31;
  const long long wid = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const long long nw = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  const long long n = a.amb[0];
  const float sc = static_cast<float>(a.sm_scale);
  for (long long qi = wid; qi < n; qi += nw) {
    const int64_t gw = a.amb[1 + qi];
    int b = 0;
    while (b + 1 < a.num_reqs && a.row_off[b + 1] <= gw) ++b;
    const ReqInfo ri = req_info(a, b);
    const int64_t local = gw - a.row_off[b];
    const int h = static_cast<int>(local / ri.R);
    const int r = static_cast<int>(local % ri.R);
    const int kvh = h / (a.num_q_heads / a.num_kv_heads);
    const int rp = (ri.R + kRowTile - 1) / kRowTile * kRowTile;
    const int qblk = r / KB;
    const float* bm_row = a.bm + a.bm_off[b] + static_cast<int64_t>(h) * bm_block_base(ri.nqb, KB) +
                          bm_block_base(qblk, KB) + (r - qblk * KB);   // block j at bm_row[j * KB]
    const float thr = a.v1[gw] - 3.0f * a.err[gw];
    float qf[PER];
    {
      const uint16_t* qrow = a.qs + (a.qs_off[b] + static_cast<int64_t>(h) * rp + r) * HD + lane * PER;
#pragma unroll
      for (int e = 0; e < PER; ++e) qf[e] = bf16_to_f32(qrow[e]);
    }
    const int64_t krow0 = a.ks_off[b] + static_cast<int64_t>(kvh) * rp;
    uint32_t* bits = a.hrm_bits + gw * a.words_per_row;
    for (int w = lane; w < a.words_per_row; w += 32) bits[w] = 0u;
    __syncwarp();
    // candidate blocks, 32 per ballot, all block maxima of a group of 1024 blocks loaded at once;
    // one pass over their keys keeps each candidate block's largest exact logit (lane k holds the
    // k-th candidate's), a second pass is taken only when there are more than 32 candidates
    double M = -INFINITY;
    double bmx_lane = -INFINITY;
    int bj_lane = -1, ncand = 0;
    for (int g0 = 0; g0 <= qblk; g0 += 1024) {
      uint32_t cmk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int j = g0 + c * 32 + lane;
        const float bmj = (j <= qblk) ? bm_row[static_cast<int64_t>(j) * KB] : -INFINITY;
        cmk[c] = __ballot_sync(0xffffffffu, bmj != -INFINITY && bmj * sc >= thr);
      }
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        uint32_t cm = cmk[c];
        while (cm) {
          const int jj = g0 + c * 32 + __ffs(cm) - 1;
          cm &= cm - 1;
          float kf[KB][PER];
          bool vis[KB];
#pragma unroll
          for (int q = 0; q < KB; ++q) {
            const int kc = jj * KB + q;
            vis[q] = kc <= r && ((a.kvalid[(krow0 + kc) >> 5] >> ((krow0 + kc) & 31)) & 1u);
            const uint16_t* kr = a.ks + (krow0 + (vis[q] ? kc : 0)) * HD + lane * PER;
#pragma unroll
            for (int e = 0; e < PER; ++e) kf[q][e] = bf16_to_f32(kr[e]);
          }
          double bx = -INFINITY;
#pragma unroll
          for (int q = 0; q < KB; ++q) {
            double part = 0.0;
#pragma unroll
            for (int e = 0; e < PER; ++e) part += static_cast<double>(qf[e] * kf[q][e]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (vis[q]) bx = fmax(bx, part * a.sm_scale);
          }
          if (lane == (ncand & 31) && ncand < 32) { bmx_lane = bx; bj_lane = jj; }
          ++ncand;
          M = fmax(M, bx);
        }
      }
    }
    if (ncand <= 32) {
      if (bj_lane >= 0 && bmx_lane == M) atomicOr(&bits[bj_lane >> 5], 1u << (bj_lane & 31));
    } else {
      for (int j0 = 0; j0 <= qblk; j0 += 32) {
        const int j = j0 + lane;
        const float bmj = (j <= qblk) ? bm_row[static_cast<int64_t>(j) * KB] : -INFINITY;
        unsigned cm = __ballot_sync(0xffffffffu, bmj != -INFINITY && bmj * sc >= thr);
        while (cm) {
          const int jj = j0 + __ffs(cm) - 1;
          cm &= cm - 1;
          bool hit = false;
          for (int q = 0; q < KB; ++q) {
            const int kc = jj * KB + q;
            if (kc > r) break;
            if (!((a.kvalid[(krow0 + kc) >> 5] >> ((krow0 + kc) & 31)) & 1u)) continue;
            const uint16_t* kr = a.ks + (krow0 + kc) * HD + lane * PER;
            double part = 0.0;
#pragma unroll
            for (int e = 0; e < PER; ++e) part += static_cast<double>(qf[e] * bf16_to_f32(kr[e]));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            hit = hit || (part * a.sm_scale == M);
          }
          if (hit && lane == 0) atomicOr(&bits[jj >> 5], 1u << (jj & 31));
        }
      }
    }
    if (lane == 0) a.M[gw] = M;
  }
}

// ---------------------------------------------------------------------------
// per query block: flag-grouped sort, certification, float64 repair, mask row
// ---------------------------------------------------------------------------
// dynamic shared memory of kap_select for `cap` candidates (a power of two)
constexpr int kRepChunk = 64;            // repaired positions per round of the float64 repair
// per warp of the select kernel: one key block staged for the bulk exact scores, rows padded by 16 bytes
// (the rows of a block then start in different banks); sized for 16 keys of d = 128
constexpr int kBulkRowPitch = 128 + 8;    // bf16 elements
constexpr size_t kBulkSlabBytes = static_cast<size_t>(kSelectThreads / 32) * 16 * kBulkRowPitch * 2;
__host__ __device__ inline size_t select_smem_bytes(int cap) {
  return static_cast<size_t>(cap) * (8 + 4 + 4 + 4 + 4 + 8 + 1 + 1) + 64 + kRepChunk * 16 * sizeof(double) + 64 +
         kBulkSlabBytes;
}

__device__ __forceinline__ unsigned long long sort_key(bool hrm, float s, int j) {
  // descending order of the key = HRM first, then score descending, then block ascending
  return (static_cast<unsigned long long>(hrm) << 63) | (static_cast<unsigned long long>(__float_as_uint(s)) << 31) |
         static_cast<unsigned long long>(0x7FFFFFFF - j);
}
__device__ __forceinline__ int key_block(unsigned long long k) { return 0x7FFFFFFF - static_cast<int>(k & 0x7FFFFFFFull); }

// ---- bitonic sort (descending) of kSelectThreads * E keys held E per thread, thread t holding
// positions t*E .. t*E+E-1: partners closer than E are swapped in registers, closer than 32*E
// through warp shuffles, the rest through shared memory.
template <int JJ, int E>
__device__ __forceinline__ void sort_stage_reg(unsigned long long (&v)[E], int k, int tid) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if ((e & JJ) == 0) {
      const int x = tid * E + e;
      const bool desc = (x & k) == 0;
      const unsigned long long lo = v[e], hi = v[e | JJ];
      const bool sw = desc ? (lo < hi) : (lo > hi);
      v[e] = sw ? hi : lo;
      v[e | JJ] = sw ? lo : hi;
    }
  }
}

template <int E>
__device__ void sort_keys_desc(unsigned long long (&v)[E], unsigned long long* buf, int N) {
  const int tid = threadIdx.x, lane = tid & 31;
  for (int k = 2; k <= N; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      if (jj < E) {
        if (jj == 1) sort_stage_reg<1, E>(v, k, tid);
        else if constexpr (E > 2) {
          if (jj == 2) sort_stage_reg<2, E>(v, k, tid);
          else if constexpr (E > 4) {
            if (jj == 4) sort_stage_reg<4, E>(v, k, tid);
            else if constexpr (E > 8) {
              if (jj == 8) sort_stage_reg<8, E>(v, k, tid);
            }
          }
        }
      } else if (jj < 32 * E) {
        const int ld = jj / E;
        const bool lower = (lane & ld) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[e], ld);
          const bool desc = ((tid * E + e) & k) == 0;
          const bool take_max = (lower == desc);
          v[e] = take_max ? (v[e] > o ? v[e] : o) : (v[e] < o ? v[e] : o);
        }
      } else {
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) buf[tid * E + e] = v[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int x = tid * E + e, y = x ^ jj;
          const unsigned long long o = buf[y];
          const bool take_max = (x < y) == ((x & k) == 0);
          v[e] = take_max ? (v[e] > o ? v[e] : o) : (v[e] < o ? v[e] : o);
        }
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < E; ++e) buf[tid * E + e] = v[e];
  __syncthreads();
}

// keys[j] for j < J (0 past J) sorted descending into key[0..N)
template <int E>
__device__ void sort_block_keys(unsigned long long* key, const uint8_t* hrm, const float* score, int J, int N) {
  unsigned long long v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = threadIdx.x * E + e;
    v[e] = (j < J) ? sort_key(hrm[j] != 0, fmaxf(score[j], 0.0f), j) : 0ull;
  }
  sort_keys_desc<E>(v, key, N);
}

constexpr int kTopFast = 128;             // budgets up to this many blocks take the top-K path

// Shared state of the top-K selection.
struct TopkShared {
  uint32_t hist[256];
  int digit, above, count;
  int hi_out[2];                          // float bits of the largest upper bound of the unselected
                                          // keys of each group ([0] rest, [1] HRM); scores are >= 0
  int warp_cnt[kSelectThreads / 32];
};

// The K largest of the J keys (distinct) into key[0..K), sorted descending, key[K..256) = 0; the largest
// upper bound (score + error) of the unselected keys of each group into sh.hi_out.  Radix select on
// 8-bit digits from the top finds the K-th key; the winners are compacted and sorted.
template <int E>
__device__ void select_top_keys(unsigned long long* key, const uint8_t* hrm, const float* score,
                                const float* serr, int J, int K, TopkShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  unsigned long long v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = tid * E + e;
    v[e] = (j < J) ? sort_key(hrm[j] != 0, fmaxf(score[j], 0.0f), j) : 0ull;
  }
  unsigned long long prefix = 0ull, pmask = 0ull;
  int krem = K;   // rank (from the top, 1-based) of the K-th key among the keys matching the prefix
  for (int shift = 56; shift >= 0; shift -= 8) {
    __syncthreads();
    for (int d = tid; d < 256; d += blockDim.x) sh.hist[d] = 0;
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (tid * E + e < J && (v[e] & pmask) == prefix) atomicAdd(&sh.hist[(v[e] >> shift) & 255u], 1u);
    __syncthreads();
    if (w == 0) {
      // lane l holds digits 255 - 8l .. 248 - 8l (highest first)
      int cq[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) { cq[q] = static_cast<int>(sh.hist[255 - 8 * lane - q]); sum += cq[q]; }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int run = incl - sum;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (run < krem && run + cq[q] >= krem) { sh.digit = 255 - 8 * lane - q; sh.above = run; sh.count = cq[q]; }
        run += cq[q];
      }
    }
    __syncthreads();
    const int d = sh.digit;
    krem -= sh.above;
    prefix |= static_cast<unsigned long long>(d) << shift;
    pmask |= 0xFFull << shift;
    if (sh.count == krem) break;   // every key with this prefix is among the K
  }
  // a key is selected iff its masked top bits are at least the prefix: exactly K keys
  int cnt = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) cnt += (tid * E + e < J && (v[e] & pmask) >= prefix) ? 1 : 0;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh.warp_cnt[w] = incl;
  if (tid < 2) sh.hi_out[tid] = __float_as_int(-INFINITY);
  key[tid] = 0ull;   // kSelectThreads slots
  __syncthreads();
  int pos = incl - cnt;
  for (int q = 0; q < w; ++q) pos += sh.warp_cnt[q];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = tid * E + e;
    if (j >= J) continue;
    if ((v[e] & pmask) >= prefix) {
      key[pos++] = v[e];
    } else {
      const float hv = fmaxf(score[j], 0.0f) + serr[j];
      atomicMax(&sh.hi_out[hrm[j] != 0 ? 1 : 0], __float_as_int(hv));
    }
  }
  __syncthreads();
  unsigned long long s1[1] = {key[tid]};
  sort_keys_desc<1>(s1, key, kSelectThreads);
}

// Top-p length (the shortest prefix of rho_i whose scores reach p of the row's total), bracketed by
// the score intervals [s - e, s + e] (s clamped at 0) of the sorted candidates key[0..J).  With
//   f(k) = (1 - p) sum_{x<k} s_x - p sum_{x>=k} s_x,
// non-decreasing in k, the exact length is the least k with f(k) >= 0: it is at least K_lo, the least
// k whose upper bound of f reaches 0, and at most K_hi, the least k whose lower bound does.  Sums in
// float64; a margin of 1e-12 of the total covers their rounding.  K_lo == K_hi certifies the length.
__device__ int2 top_p_range(const unsigned long long* key, const float* score, const float* serr, int J, int ppm,
                            double* ws_lo, double* ws_hi, int* kr) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int E = (J + kSelectThreads - 1) / kSelectThreads;
  double plo = 0.0, phi = 0.0;
  for (int e = 0; e < E; ++e) {
    const int x = tid * E + e;
    if (x >= J) break;
    const int j = key_block(key[x]);
    const float sv = fmaxf(score[j], 0.0f);
    plo += static_cast<double>(fmaxf(sv - serr[j], 0.0f));
    phi += static_cast<double>(sv) + static_cast<double>(serr[j]);
  }
  double ilo = plo, ihi = phi;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double ylo = __shfl_up_sync(0xffffffffu, ilo, o);
    const double yhi = __shfl_up_sync(0xffffffffu, ihi, o);
    if (lane >= o) {
      ilo += ylo;
      ihi += yhi;
    }
  }
  if (lane == 31) {
    ws_lo[w] = ilo;
    ws_hi[w] = ihi;
  }
  if (tid == 0) kr[0] = kr[1] = J;
  __syncthreads();
  double run_lo = ilo - plo, run_hi = ihi - phi, TL = 0.0, TH = 0.0;
  for (int q = 0; q < kSelectThreads / 32; ++q) {
    if (q < w) {
      run_lo += ws_lo[q];
      run_hi += ws_hi[q];
    }
    TL += ws_lo[q];
    TH += ws_hi[q];
  }
  const double p = static_cast<double>(ppm) / 1e6, eps = 1e-12 * TH;
  // both tests are monotone in x: each thread reports only its first position passing each
  bool got_lo = false;
  for (int e = 0; e < E; ++e) {
    const int x = tid * E + e;
    if (x >= J) break;
    const int j = key_block(key[x]);
    const float sv = fmaxf(score[j], 0.0f);
    run_lo += static_cast<double>(fmaxf(sv - serr[j], 0.0f));
    run_hi += static_cast<double>(sv) + static_cast<double>(serr[j]);
    // prefix of length x + 1: upper bound of f >= 0 possible, lower bound of f >= 0 certain
    if (!got_lo && (1.0 - p) * run_hi + p * run_lo >= p * TL - eps) {
      atomicMin(&kr[0], x + 1);
      got_lo = true;
    }
    if (got_lo && (1.0 - p) * run_lo + p * run_hi >= p * TH + eps) {
      atomicMin(&kr[1], x + 1);
      break;
    }
  }
  __syncthreads();
  int2 r = make_int2(kr[0], kr[1]);
  __syncthreads();
  r.x = r.x < 1 ? 1 : (r.x > J ? J : r.x);
  r.y = r.y < r.x ? r.x : (r.y > J ? J : r.y);
  return r;
}

template <int E>
__device__ void select_top_dispatch(unsigned long long* key, const uint8_t* hrm, const float* score,
                                    const float* serr, int J, int K, TopkShared& sh) {
  select_top_keys<E>(key, hrm, score, serr, J, K, sh);
}

// Exact scores s_ij = sum over the query block's sampled rows r (ascending) of exp(bm[r,j] - M_r) with
// float64-accurate logits, for the blocks at positions pos[0..n) of the sorted keys, into val[0..n).
// A warp per (position, row): lane group kgrp holds key j*KB + kgrp of the block, its LPK lanes split
// d; the keys whose fp32 logit lies within 2 e_r of the block's fp32 maximum get the float64 dot.
// Ends with the block synchronised.
template <int HD, int KB>
__device__ void exact_scores(const KapArgs& a, const unsigned long long* key, const int32_t* pos, int n, double* val,
                             double* terms, int b, int h, int kvh, int r0, int r1, int R, int64_t rbase) {
  constexpr int LPK = 32 / KB;
  constexpr int SL = HD / LPK;
  const int tid = threadIdx.x;
  const int warps = blockDim.x / 32, w = tid >> 5, lane = tid & 31;
  const int kgrp = lane / LPK, sub = lane % LPK;
  const int nrows = r1 - r0;
  const int rp = (R + kRowTile - 1) / kRowTile * kRowTile;
  const uint16_t* qbase = a.qs + (a.qs_off[b] + static_cast<int64_t>(h) * rp) * HD;
  const int64_t krow0 = a.ks_off[b] + static_cast<int64_t>(kvh) * rp;
  const float sc = static_cast<float>(a.sm_scale);
  for (int base = 0; base < n; base += kRepChunk) {
    const int nm = min(kRepChunk, n - base);
    for (int item = w; item < nm * nrows; item += warps) {
      const int m = base + item / nrows, r = r0 + item % nrows;
      const int j = key_block(key[pos[m]]);
      const double Mr = a.M[rbase + r];
      double term = 0.0;
      if (Mr != -INFINITY) {
        const int kc = j * KB + kgrp;
        const bool vis = kc <= r && ((a.kvalid[(krow0 + kc) >> 5] >> ((krow0 + kc) & 31)) & 1u);
        const uint16_t* qr = qbase + static_cast<int64_t>(r) * HD + sub * SL;
        // keys past the row (or past the request) are not read: their lanes use the query row
        const uint16_t* kr = vis ? a.ks + (krow0 + kc) * HD + sub * SL : qr;
        // two interleaved partial sums: rounding depth SL/2 + 1 + log2(LPK) stays within e_r
        float p0 = 0.0f, p1 = 0.0f;
#pragma unroll 1
        for (int e = 0; e < SL; e += 8) {
          float qv[8], kv[8];
          load8_bf16(qr + e, qv);
          load8_bf16(kr + e, kv);
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            p0 = fmaf(qv[i], kv[i], p0);
            p1 = fmaf(qv[i + 1], kv[i + 1], p1);
          }
        }
        float part = p0 + p1;
#pragma unroll
        for (int o = LPK / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        const float x = vis ? part * sc : -INFINITY;
        float mx = x;
#pragma unroll
        for (int o = LPK; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (mx != -INFINITY) {
          // candidates: keys whose fp32 logit is within 2 e_r of the row's block maximum; each
          // candidate's float64 logit is taken by the whole warp (four elements per lane)
          const bool cand = vis && x >= mx - 2.0f * a.err[rbase + r];
          uint32_t cmask = __ballot_sync(0xffffffffu, cand && sub == 0);
          double dv = -INFINITY;
          const uint16_t* qrow = qbase + static_cast<int64_t>(r) * HD;
          float qf[HD / 32];
#pragma unroll
          for (int e = 0; e < HD / 32; ++e) qf[e] = bf16_to_f32(qrow[lane * (HD / 32) + e]);
          while (cmask) {
            const int g = (__ffs(cmask) - 1) / LPK;   // key group of the candidate
            cmask &= cmask - 1;
            const uint16_t* krow = a.ks + (krow0 + j * KB + g) * HD;
            float kf[HD / 32];
#pragma unroll
            for (int e = 0; e < HD / 32; ++e) kf[e] = bf16_to_f32(krow[lane * (HD / 32) + e]);
            dv = fmax(dv, warp_dot3<HD / 32>(qf, kf) * a.sm_scale);   // float64 accuracy, FP32 pipe
          }
          term = dv - Mr;   // exponent; exp is taken below, one item per thread
        } else {
          term = -INFINITY;
        }
      } else {
        term = -INFINITY;
      }
      if (lane == 0) terms[item] = term;
    }
    __syncthreads();
    for (int item = tid; item < nm * nrows; item += blockDim.x) terms[item] = exp(terms[item]);
    __syncthreads();
    for (int m = tid; m < nm; m += blockDim.x) {
      double sum = 0.0;
      for (int rr = 0; rr < nrows; ++rr) sum += terms[m * nrows + rr];
      val[base + m] = sum;
    }
    __syncthreads();
  }
}

// The same exact scores for the positions [x0, x1) at once (the top-p length's exact path, which can
// need a whole row): a warp per position and every (sampled row, key) pair of its block in the warp,
// lane = (row q = lane / L, keys sub, sub + L, ...) with L = 32 / KB lanes per row.  fp32 dots with
// eight partial sums (rounding depth HD / 8 + 3 <= 19, within e_r), the row's maximum across its L
// lanes, the keys within 2 e_r of it summed as three fp32 terms by their own lanes (float64
// accuracy), rows summed in ascending order.  qrows: the query block's sampled rows, bf16, staged in
// shared memory by the caller.  Ends with the block synchronised.
template <int HD, int KB>
__device__ void exact_scores_bulk(const KapArgs& a, const unsigned long long* key, int x0, int x1, double* val,
                                  const uint16_t* qrows, uint16_t* slab, int b, int kvh, int r0, int r1, int R,
                                  int64_t rbase) {
  constexpr int L = 32 / KB;                     // lanes per sampled row
  constexpr int KPL = (KB + L - 1) / L;          // keys per lane
  constexpr int CH = HD / 8;                     // 16-byte chunks per key row
  static_assert(KB <= 16 && HD + 8 <= kBulkRowPitch, "the slab holds 16 keys of d = 128");
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, warps = blockDim.x >> 5;
  uint16_t* kb_s = slab + static_cast<size_t>(w) * 16 * kBulkRowPitch;
  const int q = lane / L, sub = lane % L;
  const int r = r0 + q;
  const bool row_ok = r < r1;
  const double Mr = row_ok ? a.M[rbase + r] : -INFINITY;
  const float er = row_ok ? a.err[rbase + r] : 0.0f;
  const int rp = (R + kRowTile - 1) / kRowTile * kRowTile;
  const int64_t krow0 = a.ks_off[b] + static_cast<int64_t>(kvh) * rp;
  const uint16_t* qrow = qrows + q * HD;
  const float sc = static_cast<float>(a.sm_scale);
  for (int x = x0 + w; x < x1; x += warps) {
    const int j = key_block(key[x]);
    // the block's KB key rows (contiguous in the gathered keys; padding rows past the request are
    // loaded but never used), one coalesced pass of the warp
    __syncwarp();
    {
      const uint4* src = reinterpret_cast<const uint4*>(a.ks + (krow0 + static_cast<int64_t>(j) * KB) * HD);
#pragma unroll
      for (int e = lane; e < KB * CH; e += 32)
        *reinterpret_cast<uint4*>(kb_s + (e / CH) * kBulkRowPitch + (e % CH) * 8) = src[e];
    }
    __syncwarp();
    float lg[KPL];
    float mx = -INFINITY;
#pragma unroll
    for (int t = 0; t < KPL; ++t) {
      const int kk = sub + L * t, kc = j * KB + kk;
      const bool vis = row_ok && kk < KB && kc <= r && ((a.kvalid[(krow0 + kc) >> 5] >> ((krow0 + kc) & 31)) & 1u);
      lg[t] = -INFINITY;
      if (vis) {
        const uint16_t* krow = kb_s + kk * kBulkRowPitch;
        float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
        for (int e = 0; e < HD; e += 8) {
          float qv[8], kv[8];
          load8_bf16(qrow + e, qv);
          load8_bf16(krow + e, kv);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(qv[i], kv[i], acc[i]);
        }
        lg[t] = (((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]))) * sc;
        mx = fmaxf(mx, lg[t]);
      }
    }
#pragma unroll
    for (int o = 1; o < L; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    double dv = -INFINITY;
#pragma unroll
    for (int t = 0; t < KPL; ++t) {
      if (lg[t] != -INFINITY && lg[t] >= mx - 2.0f * er) {
        const uint16_t* krow = kb_s + (sub + L * t) * kBulkRowPitch;
        float hi = 0.0f, lo = 0.0f, cc = 0.0f;
#pragma unroll 2
        for (int e = 0; e < HD; e += 8) {
          float qv[8], kv[8];
          load8_bf16(qrow + e, qv);
          load8_bf16(krow + e, kv);
#pragma unroll
          for (int i = 0; i < 8; ++i) sum3_add(hi, lo, cc, __fmul_rn(qv[i], kv[i]));
        }
        const double d = (static_cast<double>(hi) + static_cast<double>(lo)) + static_cast<double>(cc);
        dv = fmax(dv, d * a.sm_scale);
      }
    }
#pragma unroll
    for (int o = 1; o < L; o <<= 1) dv = fmax(dv, __shfl_xor_sync(0xffffffffu, dv, o));
    double term = 0.0;
    if (sub == 0 && Mr != -INFINITY && dv != -INFINITY) term = exp(dv - Mr);
    double sum = 0.0;
#pragma unroll
    for (int qq = 0; qq < KB; ++qq) {
      const double tq = __shfl_sync(0xffffffffu, term, qq * L);
      if (r0 + qq < r1) sum += tq;
    }
    if (lane == 0) val[x] = sum;
  }
  __syncthreads();
}

// Selection of mask row `row` by the whole block (the rows kap_select_warp_kernel leaves).
template <int HD, int KB>
__device__ void kap_select_row(const KapArgs& a, int cap, int row) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  unsigned long long* key = reinterpret_cast<unsigned long long*>(smem_raw);  // [cap] sort keys
  double* rep_val = reinterpret_cast<double*>(key + cap);                      // [cap] exact scores
  float* lo = reinterpret_cast<float*>(rep_val + cap);                         // [cap] lower bounds
  float* hi = lo + cap;                                                        // [cap] upper bounds
  float* suf = hi + cap;                                                       // [cap] suffix max of hi
  int32_t* rep_pos = reinterpret_cast<int32_t*>(suf + cap);                    // [cap] positions to repair
  uint8_t* hrm = reinterpret_cast<uint8_t*>(rep_pos + cap);                    // [cap] HRM flags
  double* terms = reinterpret_cast<double*>(
      (reinterpret_cast<uintptr_t>(hrm + 2 * cap) + 15) & ~uintptr_t(15));     // [kRepChunk * KB] row terms
  uint8_t* cutf = hrm + cap;                                                   // [cap] certain-cut flags
  __shared__ int32_t n_rep_s, n_hrm_s, cstar_s[2], warp_cnt_s[kSelectThreads / 32], sentinel_marked_s, topk_s;
  __shared__ int32_t krange_s[2], klo_s;
  __shared__ double warp_sum_s[kSelectThreads / 32], warp_sum2_s[kSelectThreads / 32];
  __shared__ TopkShared topk;

  const int tid = threadIdx.x;
  int idx = row;
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
  // K_i of the fraction rule; the top-p rule replaces it once the candidates are sorted
  int K = max(1, min(J, static_cast<int>((static_cast<long long>(a.budget_ppm) * J + 999999) / 1000000)));
  const int kvh = h / (a.num_q_heads / a.num_kv_heads);
  const int nqb = ri.nqb;
  const int64_t sbase = a.sc_off[b] + static_cast<int64_t>(h) * nqb * nqb + static_cast<int64_t>(i) * nqb;
  const int r0 = i * a.kb, r1 = min((i + 1) * a.kb, ri.R);
  const int64_t rbase = a.row_off[b] + static_cast<int64_t>(h) * ri.R;

  // HRM flags of the candidates (exact, from the float64 row maxima)
  for (int j = tid; j < J; j += blockDim.x) hrm[j] = 0;
  __syncthreads();
  if (tid < r1 - r0) {                       // one thread per sampled row of the query block
    const int r = r0 + tid;
    const int fl = a.rflags[rbase + r];
    if (fl & 1) {
      const uint32_t* bits = a.hrm_bits + (rbase + r) * a.words_per_row;
      for (int j = 0; j < J; ++j)
        if ((bits[j >> 5] >> (j & 31)) & 1u) hrm[j] = 1;
    } else if (!(fl & 2)) {
      hrm[(a.c1[rbase + r] * a.stride) / a.block_size] = 1;
    }
  }
  __syncthreads();
  if (tid == 0) n_hrm_s = 0;
  {
    int cnt = 0;
    for (int j = tid; j < J; j += blockDim.x) cnt += hrm[j] != 0;
    __syncthreads();
    if (cnt) atomicAdd(&n_hrm_s, cnt);
  }
  __syncthreads();
  const int nh_all = n_hrm_s;   // HRM keys sort first
  const float* sc = a.score + sbase;
  const float* se = a.score_err + sbase;
  // Ordered list the certification runs on: either all J keys sorted (full path), or the ks largest
  // keys sorted plus one sentinel at position ks that stands for every unselected key of its group
  // (its upper bound is theirs, largest; it is never a candidate).  The first attempt takes ks = K;
  // if the budget cut cannot be certified against that sentinel (an uncertain run reaches it), a
  // second takes ks = K + 32, so that the run can close before the sentinel; then the full path.
  int Jl = J, nh = nh_all, n2 = 1, Nl = kSelectThreads;
  int ks = K;                // selected keys (the sentinel's position) on the top-K paths
  bool sentinel = false;
  bool topp_exact = false;   // the top-p length is not certified by the bounds: exact scores below
  float sentinel_hi = -INFINITY;
  for (int attempt = (!a.top_p && K <= kTopFast && K < J) ? 0 : 2; attempt < 3; ++attempt) {
    int N2 = 1;
    while (N2 < J) N2 <<= 1;
    const int N = N2 < kSelectThreads ? kSelectThreads : N2;
    if (attempt == 1) {
      ks = min(min(K + 32, kTopFast), J - 1);
      if (ks <= K) continue;   // no room to widen: the full path
    }
    if (attempt < 2) {
      if (attempt == 0) ks = K;
      switch (N / kSelectThreads) {
        case 1: select_top_dispatch<1>(key, hrm, sc, se, J, ks, topk); break;
        case 2: select_top_dispatch<2>(key, hrm, sc, se, J, ks, topk); break;
        case 4: select_top_dispatch<4>(key, hrm, sc, se, J, ks, topk); break;
        case 8: select_top_dispatch<8>(key, hrm, sc, se, J, ks, topk); break;
        default: select_top_dispatch<16>(key, hrm, sc, se, J, ks, topk); break;
      }
      sentinel = true;
      Jl = ks + 1;
      nh = (nh_all > ks) ? ks + 1 : nh_all;   // the sentinel joins the HRM group iff HRM keys were left out
      sentinel_hi = __int_as_float(topk.hi_out[(nh_all > ks) ? 1 : 0]);
      Nl = kSelectThreads;
    } else {
      switch (N / kSelectThreads) {
        case 1: sort_block_keys<1>(key, hrm, sc, J, N); break;
        case 2: sort_block_keys<2>(key, hrm, sc, J, N); break;
        case 4: sort_block_keys<4>(key, hrm, sc, J, N); break;
        case 8: sort_block_keys<8>(key, hrm, sc, J, N); break;
        default: sort_block_keys<16>(key, hrm, sc, J, N); break;
      }
      if (a.top_p) {
        // a certified length, or every position's exact score decides it below
        const int2 kr = top_p_range(key, sc, se, J, a.budget_ppm, warp_sum_s, warp_sum2_s, krange_s);
        K = kr.y;
        topp_exact = kr.x != kr.y;
        if (tid == 0) klo_s = kr.x;
      }
      sentinel = false;
      Jl = J;
      nh = nh_all;
      Nl = N;
    }
    n2 = 1;
    while (n2 < Jl) n2 <<= 1;
    if (tid == 0) {
      cstar_s[0] = cstar_s[1] = 0x7fffffff;
      sentinel_marked_s = 0;
    }
    // score intervals per listed position
    for (int p = tid; p < n2; p += blockDim.x) {
      if (sentinel && p == ks) {
        lo[p] = -INFINITY;
        hi[p] = sentinel_hi;
      } else if (p < Jl) {
        const int j = key_block(key[p]);
        const float s = fmaxf(sc[j], 0.0f);
        const float e = se[j];
        lo[p] = s - e;
        hi[p] = s + e;
      } else {
        lo[p] = -INFINITY;
        hi[p] = -INFINITY;
      }
    }
    __syncthreads();
    // within each group (HRM positions [0, nh), the rest [nh, Jl)): suffix maximum of hi and prefix
    // minimum of lo (Hillis-Steele, log2(n2) rounds); lo is overwritten by its prefix minimum
    for (int p = tid; p < n2; p += blockDim.x) suf[p] = hi[p];
    __syncthreads();
    for (int off = 1; off < n2; off <<= 1) {
      float ts[16], tp[16];
      int cnt = 0;
      for (int p = tid; p < n2; p += blockDim.x, ++cnt) {
        const int q = p + off, r = p - off;
        const bool sq = q < n2 && ((p < nh) == (q < nh));
        const bool sr = r >= 0 && ((p < nh) == (r < nh));
        ts[cnt & 15] = sq ? fmaxf(suf[p], suf[q]) : suf[p];
        tp[cnt & 15] = sr ? fminf(lo[p], lo[r]) : lo[p];
      }
      __syncthreads();
      cnt = 0;
      for (int p = tid; p < n2; p += blockDim.x, ++cnt) {
        suf[p] = ts[cnt & 15];
        lo[p] = tp[cnt & 15];
      }
      __syncthreads();
    }
    // Clusters of positions whose relative order, or side of the budget cut, the bounds cannot
    // certify.  The cut after position q is certain iff every element up to q (in its group)
    // stays above every later one: min lo[g0..q] > max hi[q+1..g1).  (Cuts certified for the
    // elements of q's own run suffice: an earlier certain cut already puts all elements before
    // it above everything after it.)  Runs of two or more positions between certain cuts are
    // repaired when they start before K.
    for (int p = tid; p < Jl; p += blockDim.x) {
      const int g1 = p < nh ? nh : Jl;
      cutf[p] = (p == g1 - 1) || (lo[p] > suf[p + 1]);
    }
    __syncthreads();
    for (int p = tid; p < Jl; p += blockDim.x) {
      const int g = p < nh ? 0 : 1;
      const int g1 = g ? Jl : nh;
      const int kg = min(K, g1);
      if (p >= kg - 1 && cutf[p]) atomicMin(&cstar_s[g], p);
    }
    __syncthreads();
    {
      // each thread marks positions tid*E .. tid*E+E-1 in order; a block scan places them
      const int E = Nl / kSelectThreads;
      int cnt = 0;
      uint32_t bits = 0;
      for (int e = 0; e < E; ++e) {
        const int x = tid * E + e;
        if (x >= Jl) break;
        const int g = x < nh ? 0 : 1;
        const int g0 = g ? nh : 0, g1 = g ? Jl : nh;
        const int kg = min(K, g1);
        bool mk = false;
        if (kg > g0) {
          const bool multi = !cutf[x] || (x > g0 && !cutf[x - 1]);
          mk = multi && (x < kg || x <= cstar_s[g]);
        }
        if (mk) {
          bits |= 1u << e;
          ++cnt;
          if (sentinel && x == ks) sentinel_marked_s = 1;
        }
      }
      const int lane = tid & 31, w = tid >> 5;
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) warp_cnt_s[w] = incl;
      __syncthreads();
      int base = 0, total = 0;
      for (int q = 0; q < kSelectThreads / 32; ++q) {
        if (q < w) base += warp_cnt_s[q];
        total += warp_cnt_s[q];
      }
      int pos = base + incl - cnt;
      for (int e = 0; e < E; ++e)
        if ((bits >> e) & 1u) rep_pos[pos++] = tid * E + e;
      if (tid == 0) n_rep_s = total;
    }
    __syncthreads();
    if (!sentinel_marked_s) break;   // certified (or the full path): done
    __syncthreads();
  }
  __syncthreads();
  const int n_rep = n_rep_s;
  if (n_rep > 0) {
    exact_scores<HD, KB>(a, key, rep_pos, n_rep, rep_val, terms, b, h, kvh, r0, r1, ri.R, rbase);
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
  if (topp_exact) {
    // The score bounds leave the top-p length between klo and K (= the upper end, whose cut and the
    // order before it are certified above).  Exact scores for a prefix of the positions (which holds
    // most of the row's mass, hence most of the bounds' width), bounds for the rest: f(k) is then known
    // to within p times the rest's width.  While that leaves the sign of f open somewhere in
    // [klo, K], the exact prefix grows (K + 16 positions, then four times as many, then the row);
    // with the whole row exact, the length is the oracle's: exact scores summed in order.
    // the query block's sampled rows, bf16, in the (here unused) repair term buffer; the key slabs after it
    uint16_t* qrows = reinterpret_cast<uint16_t*>(terms);
    uint16_t* slab = reinterpret_cast<uint16_t*>(terms + kRepChunk * 16);
    {
      const int rp = (ri.R + kRowTile - 1) / kRowTile * kRowTile;
      const uint4* src = reinterpret_cast<const uint4*>(a.qs + (a.qs_off[b] + static_cast<int64_t>(h) * rp +
                                                                static_cast<int64_t>(r0)) * HD);
      for (int e = tid; e < (r1 - r0) * HD / 8; e += blockDim.x) reinterpret_cast<uint4*>(qrows)[e] = src[e];
    }
    __syncthreads();
    const double p = static_cast<double>(a.budget_ppm) / 1e6;
    int done = 0;   // exact scores of positions [0, done)
    int want = min(J, K + 16);
    while (true) {
      exact_scores_bulk<HD, KB>(a, key, done, want, rep_val, qrows, slab, b, kvh, r0, r1, ri.R, rbase);
      done = want;
      double tlo = 0.0, thi = 0.0;
      for (int x = done + tid; x < J; x += blockDim.x) {
        const int j = key_block(key[x]);
        const float sv = fmaxf(sc[j], 0.0f);
        tlo += static_cast<double>(fmaxf(sv - se[j], 0.0f));
        thi += static_cast<double>(sv) + static_cast<double>(se[j]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        tlo += __shfl_xor_sync(0xffffffffu, tlo, o);
        thi += __shfl_xor_sync(0xffffffffu, thi, o);
      }
      if ((tid & 31) == 0) {
        warp_sum_s[tid >> 5] = tlo;
        warp_sum2_s[tid >> 5] = thi;
      }
      __syncthreads();
      if (tid == 0) {
        if (done == J) {
          // every score exact: summed in order, as the scores of Eq. (11) are summed for the cut
          double tot = 0.0;
          for (int x = 0; x < J; ++x) tot += rep_val[x];
          const double thr = p * tot;
          double run = 0.0;
          int k = J;
          for (int x = 0; x < J; ++x) {
            run += rep_val[x];
            if (run >= thr) {
              k = x + 1;
              break;
            }
          }
          topk_s = k < K ? k : K;
        } else {
          double TLo = 0.0, THi = 0.0, pre = 0.0;
          for (int q = 0; q < kSelectThreads / 32; ++q) {
            TLo += warp_sum_s[q];
            THi += warp_sum2_s[q];
          }
          for (int x = 0; x < done; ++x) pre += rep_val[x];
          const double eps = 1e-12 * (pre + THi);
          int kstar = -1;
          double E = 0.0;
          for (int x = 0; x < klo_s - 1; ++x) E += rep_val[x];
          for (int k = klo_s; k <= K; ++k) {
            E += rep_val[k - 1];                        // sum of the first k exact scores
            const double Rp = pre - E;                   // exact scores of positions [k, done)
            if ((1.0 - p) * E - p * (Rp + TLo) < -eps) continue;   // f(k) < 0 for sure
            if ((1.0 - p) * E - p * (Rp + THi) >= eps) kstar = k;  // f(k) >= 0 for sure
            break;
          }
          topk_s = kstar;
        }
      }
      __syncthreads();
      if (topk_s >= 0) break;
      want = (done * 4 < J) ? done * 4 : J;
      __syncthreads();
    }
    K = topk_s;
    __syncthreads();
  }
  if (a.ascending) {
    // the same K_i blocks in ascending block order (visiting without remapping): mark them in
    // hrm[] (no longer needed), then compact the marks with a block scan
    __syncthreads();
    for (int j = tid; j < J; j += blockDim.x) hrm[j] = 0;
    __syncthreads();
    for (int k = tid; k < K; k += blockDim.x) hrm[key_block(key[k])] = 1;
    __syncthreads();
    const int E = (J + kSelectThreads - 1) / kSelectThreads;
    const int lane = tid & 31, w = tid >> 5;
    int cnt = 0;
    for (int e = 0; e < E; ++e) {
      const int j = tid * E + e;
      if (j < J && hrm[j]) ++cnt;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_cnt_s[w] = incl;
    __syncthreads();
    int pos = incl - cnt;
    for (int q = 0; q < w; ++q) pos += warp_cnt_s[q];
    for (int e = 0; e < E; ++e) {
      const int j = tid * E + e;
      if (j < J && hrm[j]) out[pos++] = j;
    }
    for (int k = K + tid; k < a.mask_pitch; k += blockDim.x) out[k] = -1;
  } else {
    for (int k = tid; k < a.mask_pitch; k += blockDim.x) out[k] = (k < K) ? key_block(key[k]) : -1;
  }
  if (tid == 0) a.mask_len[mrow] = K;
}


// ---------------------------------------------------------------------------
// The same selection, one warp per mask row, for the common rows: fraction budget, J <= 1024,
// K <= 128 and K < J.  The row's scores are staged in shared memory once; the K largest keys are
// found by radix select, sorted, certified against one sentinel standing for every unselected key
// (as in kap_select_kernel's top-K path) and up to kWarpRepMax uncertain positions are repaired at
// float64 accuracy.  Every other row (and a row whose cut the sentinel cannot certify) is left to
// kap_select_kernel, marked by mask_len = -1.
// ---------------------------------------------------------------------------
__device__ __forceinline__ size_t mrow_of(const KapArgs& a, int row) {
  const int h = row % a.num_q_heads;
  row /= a.num_q_heads;
  const int b = row % a.num_reqs;
  const int i = a.nqb_max - 1 - row / a.num_reqs;
  return (static_cast<size_t>(b) * a.num_q_heads + h) * a.nqb_max + i;
}

constexpr int kWarpSelMaxJ = 1024;
constexpr int kWarpSelMaxK = 128;
constexpr int kWarpRepMax = 16;
constexpr int kWarpSelWarps = 4;

constexpr int kWarpCand = 64;            // float64-accuracy candidates of a row's repairs (more: block kernel)
constexpr int kStageUnroll = 8;          // candidates a lane loads at once

// Shared state of one warp.  Regions whose uses do not overlap in time share storage: the candidate
// words live until the certification, the repair's buffers after it; the radix histogram until the
// compaction, the selected keys from it on.
template <int HD, int KB>
struct __align__(16) WarpSelSmem {
  union {
    uint32_t word[kWarpSelMaxJ];          // candidate j: HRM flag (bit 31) | fp32 bits of max(score, 0);
                                          // from the compaction on, a selected one's error bound
    struct {
      float4 qrows[KB * HD / 4];          // the query block's sampled rows, widened to fp32: see q_chunk
      double terms[kWarpRepMax * KB];     // (repaired position, sampled row): block maxima, then terms
      uint32_t cand[kWarpCand];           // float64-accuracy candidates: (item << 16) | key
    } rep;
  } u;
  union {
    uint32_t hist[256];                   // radix select
    unsigned long long key[kWarpSelMaxK]; // the selected keys, sorted descending
  } v;
  double rep_val[kWarpRepMax];
  int32_t rep_pos[kWarpRepMax];
};

// Index of the four fp32 elements 4c .. 4c+3 of segment seg (of LPK segments of HD / LPK elements)
// of sampled row rr in the repair's query rows: the same chunk of the LPK segments side by side, so
// LPK lanes reading one chunk of their own segments hit distinct banks.
template <int HD, int LPK>
__device__ __forceinline__ int q_chunk(int rr, int seg, int c) {
  return rr * (HD / 4) + c * LPK + seg;
}

// The radix key of candidate j: its word above the block index's complement, 63 bits in the order
// of sort_key (HRM first, score descending, block ascending); sort_key moves the HRM bit to bit 63.
__device__ __forceinline__ unsigned long long radix_key(uint32_t w, int j) {
  return (static_cast<unsigned long long>(w) << 31) | static_cast<unsigned long long>(0x7FFFFFFF - j);
}
__device__ __forceinline__ unsigned long long sort_key_of_radix(unsigned long long k) {
  return (k & ~(1ull << 62)) | ((k >> 62) << 63);
}
// the 8-bit digit of k whose lowest bit is bit `shift` (bits below 0 read as zero)
__device__ __forceinline__ uint32_t radix_digit(unsigned long long k, int shift) {
  return static_cast<uint32_t>((shift >= 0 ? (k >> shift) : (k << -shift)) & 255u);
}
__device__ __forceinline__ unsigned long long radix_bits(unsigned long long d, int shift) {
  return shift >= 0 ? (d << shift) : (d >> -shift);
}

// bitonic sort (descending) of 32 * E keys held E per lane, lane l holding positions l*E .. l*E+E-1
template <int E>
__device__ __forceinline__ void warp_sort_desc(unsigned long long (&v)[E], int lane) {
#pragma unroll 1
  for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll 1
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      if (jj < E) {
        if (jj == 1) sort_stage_reg<1, E>(v, k, lane);
        else if constexpr (E > 2) {
          if (jj == 2) sort_stage_reg<2, E>(v, k, lane);
        }
      } else {
        const int ld = jj / E;
        const bool lower = (lane & ld) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[e], ld);
          const bool desc = ((lane * E + e) & k) == 0;
          const bool take_max = (lower == desc);
          v[e] = take_max ? (v[e] > o ? v[e] : o) : (v[e] < o ? v[e] : o);
        }
      }
    }
  }
}

template <int E>
__device__ __forceinline__ void warp_sort_keys(unsigned long long* key, int K, int lane) {
  unsigned long long v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = (lane * E + e < K) ? key[lane * E + e] : 0ull;
  __syncwarp();
  warp_sort_desc<E>(v, lane);
#pragma unroll
  for (int e = 0; e < E; ++e) key[lane * E + e] = v[e];
  __syncwarp();
}

__device__ __forceinline__ float warp_max_f(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ int warp_min_i(int x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = min(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// exclusive prefix sum over the lanes
__device__ __forceinline__ int warp_excl_sum(int x, int lane) {
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  return incl - x;
}

template <int HD, int KB>
__global__ void __launch_bounds__(kWarpSelWarps * 32, 8) kap_select_warp_kernel(KapArgs a) {
  __shared__ WarpSelSmem<HD, KB> wsm[kWarpSelWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  WarpSelSmem<HD, KB>& sm = wsm[w];
  const long long nrow_all = static_cast<long long>(a.num_reqs) * a.num_q_heads * a.nqb_max;
  long long idx = static_cast<long long>(blockIdx.x) * kWarpSelWarps + w;
  if (idx >= nrow_all) return;
  const int row = static_cast<int>(idx);
  // rows left to kap_select_kernel: mask_len = -1 until it writes them
  auto defer = [&]() {
    if (lane == 0) {
      a.mask_len[mrow_of(a, row)] = -1;
      a.defer[1 + atomicAdd(&a.defer[0], 1)] = row;
    }
  };
  // the row order of kap_select_kernel: heads fastest, then requests, heaviest query blocks first
  const int h = static_cast<int>(idx % a.num_q_heads);
  idx /= a.num_q_heads;
  const int b = static_cast<int>(idx % a.num_reqs);
  const int i = a.nqb_max - 1 - static_cast<int>(idx / a.num_reqs);
  const ReqInfo ri = req_info(a, b);
  const size_t mrow = (static_cast<size_t>(b) * a.num_q_heads + h) * a.nqb_max + i;
  int32_t* out = a.mask + mrow * a.mask_pitch;
  if (i >= ri.nqb) {
    for (int k = lane; k < a.mask_pitch; k += 32) out[k] = -1;
    if (lane == 0) a.mask_len[mrow] = 0;
    return;
  }
  const int J = i + 1;
  const int K = max(1, min(J, static_cast<int>((static_cast<long long>(a.budget_ppm) * J + 999999) / 1000000)));
  if (a.top_p || a.ascending || J > kWarpSelMaxJ || K > kWarpSelMaxK || K >= J) {
    defer();
    return;
  }
  const int kvh = h / (a.num_q_heads / a.num_kv_heads);
  const int nqb = ri.nqb;
  const int64_t sbase = a.sc_off[b] + static_cast<int64_t>(h) * nqb * nqb + static_cast<int64_t>(i) * nqb;
  const float* sc = a.score + sbase;
  const float* se = a.score_err + sbase;
  const int r0 = i * a.kb, r1 = min((i + 1) * a.kb, ri.R);
  const int nrows = r1 - r0;
  const int64_t rbase = a.row_off[b] + static_cast<int64_t>(h) * ri.R;

  // Candidate words in shared memory: every score requested at once (kStageUnroll per lane in
  // flight), with the row flags and arg maxima of the query block's sampled rows; the bits all
  // radix keys share are gathered on the way (words and block-index complements are disjoint fields)
  int fl = 2, cmax = 0;
  if (lane < nrows) {
    fl = a.rflags[rbase + r0 + lane];
    cmax = a.c1[rbase + r0 + lane];
  }
  uint32_t wor = 0u, wand = 0x7FFFFFFFu, ior = 0u, iand = 0x7FFFFFFFu;
  for (int j0 = 0; j0 < J; j0 += 32 * kStageUnroll) {
    float sv[kStageUnroll];
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) {
      const int j = j0 + 32 * u + lane;
      sv[u] = (j < J) ? __ldg(sc + j) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) {
      const int j = j0 + 32 * u + lane;
      if (j < J) {
        const uint32_t wd = __float_as_uint(fmaxf(sv[u], 0.0f)) & 0x7FFFFFFFu;
        sm.u.word[j] = wd;
        wor |= wd;
        wand &= wd;
        ior |= static_cast<uint32_t>(0x7FFFFFFF - j);
        iand &= static_cast<uint32_t>(0x7FFFFFFF - j);
      }
    }
  }
  __syncwarp();
  // HRM flags (exact, from the float64 row maxima): the blocks of the keys attaining each row's
  // maximum; a block counts once, for the lane whose atomic sets its flag
  int nh_part = 0;
  if (fl & 1) {
    const uint32_t* bits = a.hrm_bits + (rbase + r0 + lane) * a.words_per_row;
    for (int q = 0; q < (J + 31) / 32; ++q) {
      uint32_t bw = bits[q];
      while (bw) {
        const int j = q * 32 + __ffs(bw) - 1;
        bw &= bw - 1;
        if (j < J) nh_part += (atomicOr(&sm.u.word[j], 0x80000000u) >> 31) ^ 1u;
      }
    }
  } else if (!(fl & 2)) {
    nh_part += (atomicOr(&sm.u.word[(cmax * a.stride) / a.block_size], 0x80000000u) >> 31) ^ 1u;
  }
  const int nh_all = __reduce_add_sync(0xffffffffu, nh_part);
  __syncwarp();
  wor = __reduce_or_sync(0xffffffffu, wor) | (nh_all > 0 ? 0x80000000u : 0u);
  wand = __reduce_and_sync(0xffffffffu, wand) | (nh_all == J ? 0x80000000u : 0u);
  ior = __reduce_or_sync(0xffffffffu, ior);
  iand = __reduce_and_sync(0xffffffffu, iand);
  const unsigned long long kor = (static_cast<unsigned long long>(wor) << 31) | ior;     // OR of every radix key
  const unsigned long long kand = (static_cast<unsigned long long>(wand) << 31) | iand;  // AND of every radix key
  const int top = 63 - __clzll(kor ^ kand);   // highest bit on which two keys differ (J >= 2 distinct keys)

  // radix select of the K largest keys on 8-bit digits, from the highest differing bit down
  unsigned long long pmask = (top >= 62) ? 0ull : ~((2ull << top) - 1ull);
  unsigned long long prefix = kand & pmask;
  int krem = K;
#pragma unroll 1
  for (int shift = top - 7; shift > -8; shift -= 8) {
    for (int d = lane; d < 256; d += 32) sm.v.hist[d] = 0u;
    __syncwarp();
    if (shift >= 31) {
      // digit and prefix within the words (the common case: scores differ)
      const uint32_t pw = static_cast<uint32_t>(prefix >> 31), mw = static_cast<uint32_t>(pmask >> 31);
      const int sw = shift - 31;
#pragma unroll 4
      for (int j = lane; j < J; j += 32) {
        const uint32_t wd = sm.u.word[j];
        if ((wd & mw) == pw) atomicAdd(&sm.v.hist[(wd >> sw) & 255u], 1u);
      }
    } else {
#pragma unroll 4
      for (int j = lane; j < J; j += 32) {
        const unsigned long long kv = radix_key(sm.u.word[j], j);
        if ((kv & pmask) == prefix) atomicAdd(&sm.v.hist[radix_digit(kv, shift)], 1u);
      }
    }
    __syncwarp();
    // lane l holds digits 255 - 8l .. 248 - 8l (highest first)
    int cq[8], sum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) { cq[q] = static_cast<int>(sm.v.hist[255 - 8 * lane - q]); sum += cq[q]; }
    int run = warp_excl_sum(sum, lane);
    int dg = -1, ab = 0, ct = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (run < krem && run + cq[q] >= krem) { dg = 255 - 8 * lane - q; ab = run; ct = cq[q]; }
      run += cq[q];
    }
    const int src = __ffs(__ballot_sync(0xffffffffu, dg >= 0)) - 1;
    dg = __shfl_sync(0xffffffffu, dg, src);
    ab = __shfl_sync(0xffffffffu, ab, src);
    ct = __shfl_sync(0xffffffffu, ct, src);
    krem -= ab;
    prefix |= radix_bits(static_cast<unsigned long long>(dg), shift);
    pmask |= radix_bits(0xFFull, shift);
    __syncwarp();
    if (ct == krem) break;   // every key with this prefix is among the K
  }
  // one pass: the K winners compacted (ballot positions), their words replaced by their error bounds
  // (the score stays in the key), and the largest upper bound of the unselected keys of each group;
  // the error bounds requested kStageUnroll at a time
  float hiR = -INFINITY, hiH = -INFINITY;
  {
    int base = 0;
    for (int j0 = 0; j0 < J; j0 += 32 * kStageUnroll) {
      uint32_t wv[kStageUnroll];
      float ev[kStageUnroll];
#pragma unroll
      for (int u = 0; u < kStageUnroll; ++u) {
        const int j = j0 + 32 * u + lane;
        wv[u] = (j < J) ? sm.u.word[j] : 0u;
        ev[u] = (j < J) ? __ldg(se + j) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < kStageUnroll; ++u) {
        const int j = j0 + 32 * u + lane;
        const unsigned long long kv = radix_key(wv[u], j);
        const bool sel = (j < J) && ((kv & pmask) >= prefix);
        const unsigned m = __ballot_sync(0xffffffffu, sel);
        if (sel) {
          sm.v.key[base + __popc(m & ((1u << lane) - 1u))] = sort_key_of_radix(kv);
          sm.u.word[j] = __float_as_uint(ev[u]);
        } else if (j < J) {
          const float hv = __uint_as_float(wv[u] & 0x7FFFFFFFu) + ev[u];
          if (wv[u] >> 31) hiH = fmaxf(hiH, hv);
          else hiR = fmaxf(hiR, hv);
        }
        base += __popc(m);
      }
    }
  }
  hiR = warp_max_f(hiR);
  hiH = warp_max_f(hiH);
  __syncwarp();
  if (K <= 32) warp_sort_keys<1>(sm.v.key, K, lane);
  else if (K <= 64) warp_sort_keys<2>(sm.v.key, K, lane);
  else warp_sort_keys<4>(sm.v.key, K, lane);

  // certification over K + 1 positions: the K keys, then one sentinel with the unselected keys'
  // largest upper bound (in the HRM group iff HRM keys were left out)
  const int Jl = K + 1;
  const int nh = (nh_all > K) ? K + 1 : nh_all;
  const float sentinel_hi = (nh_all > K) ? hiH : hiR;
  constexpr int E3 = (kWarpSelMaxK + 1 + 31) / 32;
  float lo[E3], hi[E3];
#pragma unroll
  for (int e = 0; e < E3; ++e) {
    const int p = lane * E3 + e;
    if (p == K) {
      lo[e] = -INFINITY;
      hi[e] = sentinel_hi;
    } else if (p < K) {
      const unsigned long long kp = sm.v.key[p];
      const float s = __uint_as_float(static_cast<uint32_t>(kp >> 31) & 0x7FFFFFFFu);
      const float er = __uint_as_float(sm.u.word[key_block(kp)]);
      lo[e] = s - er;
      hi[e] = s + er;
    } else {
      lo[e] = -INFINITY;
      hi[e] = -INFINITY;
    }
  }
  // within each group: suffix maximum of hi and prefix minimum of lo
  float suf[E3], pre[E3];
  {
    float sH[E3], sR[E3], pH[E3], pR[E3];
    float aH = -INFINITY, aR = -INFINITY;
#pragma unroll
    for (int e = E3 - 1; e >= 0; --e) {
      const int p = lane * E3 + e;
      aH = fmaxf(aH, p < nh ? hi[e] : -INFINITY);
      aR = fmaxf(aR, p >= nh ? hi[e] : -INFINITY);
      sH[e] = aH;
      sR[e] = aR;
    }
    float bH = INFINITY, bR = INFINITY;
#pragma unroll
    for (int e = 0; e < E3; ++e) {
      const int p = lane * E3 + e;
      bH = fminf(bH, p < nh ? lo[e] : INFINITY);
      bR = fminf(bR, p >= nh ? lo[e] : INFINITY);
      pH[e] = bH;
      pR[e] = bR;
    }
    // lanes after this one (suffix) and before it (prefix)
    float xH = aH, xR = aR, yH = bH, yR = bR;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float tH = __shfl_down_sync(0xffffffffu, xH, o), tR = __shfl_down_sync(0xffffffffu, xR, o);
      const float uH = __shfl_up_sync(0xffffffffu, yH, o), uR = __shfl_up_sync(0xffffffffu, yR, o);
      if (lane + o < 32) { xH = fmaxf(xH, tH); xR = fmaxf(xR, tR); }
      if (lane >= o) { yH = fminf(yH, uH); yR = fminf(yR, uR); }
    }
    float nxH = __shfl_down_sync(0xffffffffu, xH, 1), nxR = __shfl_down_sync(0xffffffffu, xR, 1);
    float pvH = __shfl_up_sync(0xffffffffu, yH, 1), pvR = __shfl_up_sync(0xffffffffu, yR, 1);
    if (lane == 31) { nxH = -INFINITY; nxR = -INFINITY; }
    if (lane == 0) { pvH = INFINITY; pvR = INFINITY; }
#pragma unroll
    for (int e = 0; e < E3; ++e) {
      const int p = lane * E3 + e;
      suf[e] = (p < nh) ? fmaxf(sH[e], nxH) : fmaxf(sR[e], nxR);
      pre[e] = (p < nh) ? fminf(pH[e], pvH) : fminf(pR[e], pvR);
    }
  }
  // the cut after position p is certain iff everything up to p (in its group) stays above
  // everything after it
  bool cutf[E3];
  {
    const float suf_next_lane = __shfl_down_sync(0xffffffffu, suf[0], 1);
#pragma unroll
    for (int e = 0; e < E3; ++e) {
      const int p = lane * E3 + e;
      const int g1 = p < nh ? nh : Jl;
      const float sn = (e + 1 < E3) ? suf[(e + 1 < E3) ? e + 1 : e] : suf_next_lane;
      cutf[e] = (p < Jl) && ((p == g1 - 1) || (pre[e] > sn));
    }
  }
  int cs0 = 0x7fffffff, cs1 = 0x7fffffff;
#pragma unroll
  for (int e = 0; e < E3; ++e) {
    const int p = lane * E3 + e;
    if (p >= Jl || !cutf[e]) continue;
    const int g = p < nh ? 0 : 1;
    const int g1 = g ? Jl : nh;
    if (p >= min(K, g1) - 1) {
      if (g) cs1 = min(cs1, p);
      else cs0 = min(cs0, p);
    }
  }
  cs0 = warp_min_i(cs0);
  cs1 = warp_min_i(cs1);
  // positions to repair: runs of two or more between certain cuts that start before the cut
  bool mk[E3];
  int nmk = 0;
  bool sentinel_marked = false;
  {
    const bool prev_cut_lane = __shfl_up_sync(0xffffffffu, cutf[E3 - 1], 1);
#pragma unroll
    for (int e = 0; e < E3; ++e) {
      const int x = lane * E3 + e;
      mk[e] = false;
      if (x >= Jl) continue;
      const int g = x < nh ? 0 : 1;
      const int g0 = g ? nh : 0, g1 = g ? Jl : nh;
      const int kg = min(K, g1);
      if (kg > g0) {
        const bool prev_cut = (e > 0) ? cutf[(e > 0) ? e - 1 : 0] : prev_cut_lane;
        const bool multi = !cutf[e] || (x > g0 && !prev_cut);
        mk[e] = multi && (x < kg || x <= (g ? cs1 : cs0));
      }
      if (mk[e]) {
        ++nmk;
        if (x == K) sentinel_marked = true;
      }
    }
  }
  const int n_rep = __reduce_add_sync(0xffffffffu, nmk);
  if (__any_sync(0xffffffffu, sentinel_marked) || n_rep > kWarpRepMax) {
    defer();
    return;
  }
  if (n_rep > 0) {
    {
      int pos = warp_excl_sum(nmk, lane);
#pragma unroll
      for (int e = 0; e < E3; ++e)
        if (mk[e]) sm.rep_pos[pos++] = lane * E3 + e;
    }
    // exact scores s_ij = sum over rows r (ascending) of exp(bm[r,j] - M_r), bm[r, j] the largest
    // float64-accurate logit of block j for row r.  Items are (repaired position, sampled row) pairs:
    // (1) the fp32 logits of every item's keys; only keys within 2 e_r of their item's fp32 maximum
    // can attain the exact block maximum and are listed; (2) the listed candidates get logits summed
    // as three fp32 terms (float64 accuracy), four lanes each, eight candidates at a time; (3) per
    // item the largest is bm[r, j].  The candidate words are dead from here on: their storage takes
    // the query block's sampled rows, and lane rr holds row rr's M_r and e_r.
    const int n_items = n_rep * nrows;
    const int rp = (ri.R + kRowTile - 1) / kRowTile * kRowTile;
    const uint16_t* qbase = a.qs + (a.qs_off[b] + static_cast<int64_t>(h) * rp) * HD;
    const int64_t krow0 = a.ks_off[b] + static_cast<int64_t>(kvh) * rp;
    const float scl = static_cast<float>(a.sm_scale);
    double m_lane = -INFINITY;
    float e_lane = 0.0f;
    if (lane < nrows) {
      m_lane = a.M[rbase + r0 + lane];
      e_lane = a.err[rbase + r0 + lane];
    }
    __syncwarp();   // every lane's certification reads of the candidate words are done
    constexpr int LPK = 32 / KB;
    constexpr int SL = HD / LPK;
    {
      const uint16_t* src = qbase + static_cast<int64_t>(r0) * HD;
      for (int e = lane; e < nrows * HD / 8; e += 32) {
        float f[8];
        load8_bf16(src + 8 * e, f);
        const int rr = e / (HD / 8), x = 8 * (e % (HD / 8));
        const int seg = x / SL, c = (x % SL) / 4;
        sm.u.rep.qrows[q_chunk<HD, LPK>(rr, seg, c)] = make_float4(f[0], f[1], f[2], f[3]);
        sm.u.rep.qrows[q_chunk<HD, LPK>(rr, seg, c + 1)] = make_float4(f[4], f[5], f[6], f[7]);
      }
    }
    __syncwarp();
    // (1) per repaired position, the fp32 logits of the query block's sampled rows against the block's
    // sampled keys: lane group kq (LPK lanes splitting d) keeps key j*KB + kq in registers and takes
    // the rows one after another (two interleaved partial sums: rounding depth SL/2 + 1 + log2(LPK),
    // within e_r); each key row is loaded once per position
    const int kq = lane / LPK, sub = lane % LPK;
    int ncand = 0;
    for (int m = 0; m < n_rep; ++m) {
      const int kc = key_block(sm.v.key[sm.rep_pos[m]]) * KB + kq;
      const bool kvis = (a.kvalid[(krow0 + kc) >> 5] >> ((krow0 + kc) & 31)) & 1u;
      float kf[SL];
      {
        const uint16_t* kr = a.ks + (krow0 + kc) * HD + sub * SL;   // padded rows: always in the array
#pragma unroll
        for (int e = 0; e < SL; e += 8) {
          float t8[8];
          load8_bf16(kr + e, t8);
#pragma unroll
          for (int u = 0; u < 8; ++u) kf[e + u] = t8[u];
        }
      }
      for (int rr = 0; rr < nrows; ++rr) {
        const int r = r0 + rr, item = m * nrows + rr;
        const double m_r = __shfl_sync(0xffffffffu, m_lane, rr);
        const float e_r = __shfl_sync(0xffffffffu, e_lane, rr);
        const bool vis = kvis && kc <= r && m_r != -INFINITY;
        float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
        for (int e = 0; e < SL; e += 4) {
          const float4 qv = sm.u.rep.qrows[q_chunk<HD, LPK>(rr, sub, e / 4)];
          p0 = fmaf(qv.x, kf[e], p0);
          p1 = fmaf(qv.y, kf[e + 1], p1);
          p0 = fmaf(qv.z, kf[e + 2], p0);
          p1 = fmaf(qv.w, kf[e + 3], p1);
        }
        float part = p0 + p1;
#pragma unroll
        for (int o = LPK / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        const float x = vis ? part * scl : -INFINITY;
        float mx = x;
#pragma unroll
        for (int o = LPK; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const bool cand = vis && sub == 0 && x >= mx - 2.0f * e_r;
        if (lane == 0) sm.u.rep.terms[item] = -INFINITY;
        const unsigned cb = __ballot_sync(0xffffffffu, cand);
        const int slot = ncand + __popc(cb & ((1u << lane) - 1u));
        if (cand && slot < kWarpCand) sm.u.rep.cand[slot] = (static_cast<uint32_t>(item) << 16) | static_cast<uint32_t>(kc);
        ncand += __popc(cb);
      }
    }
    if (ncand > kWarpCand) {   // a row with many tied keys: the block kernel settles it
      defer();
      return;
    }
    __syncwarp();
    // (2) products of two bf16 values are exact in fp32; each candidate's sum is kept as three fp32
    // terms on the FP32 pipe (GB300's FP64 pipe runs at a small fraction of that rate)
    for (int c0 = 0; c0 < ncand; c0 += 8) {
      const int ci = c0 + lane / 4, sub4 = lane % 4;
      int item = -1;
      float shi = 0.0f, slo = 0.0f, scc = 0.0f;
      if (ci < ncand) {
        const uint32_t cw = sm.u.rep.cand[ci];
        item = static_cast<int>(cw >> 16);
        const int kc = static_cast<int>(cw & 0xffffu);
        const int rr = item % nrows;
        const uint16_t* krow = a.ks + (krow0 + kc) * HD + sub4 * (HD / 4);
#pragma unroll
        for (int e = 0; e < HD / 4; e += 8) {
          float kv[8];
          load8_bf16(krow + e, kv);
          const int x = sub4 * (HD / 4) + e;   // 8 elements within one segment (SL is a multiple of 8)
          const float4 q0 = sm.u.rep.qrows[q_chunk<HD, LPK>(rr, x / SL, (x % SL) / 4)];
          const float4 q1 = sm.u.rep.qrows[q_chunk<HD, LPK>(rr, x / SL, (x % SL) / 4 + 1)];
          const float qv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
          for (int u = 0; u < 8; ++u) sum3_add(shi, slo, scc, __fmul_rn(qv[u], kv[u]));
        }
      }
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, shi, o), ol = __shfl_xor_sync(0xffffffffu, slo, o);
        const float oc = __shfl_xor_sync(0xffffffffu, scc, o);
        sum3_add(shi, slo, scc, oh, ol, oc);
      }
      const double lx = ((static_cast<double>(shi) + static_cast<double>(slo)) + static_cast<double>(scc)) * a.sm_scale;
      // fold the round's candidates into their items' maxima, one after another
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const double v = __shfl_sync(0xffffffffu, lx, 4 * t);
        const int it = __shfl_sync(0xffffffffu, item, 4 * t);
        if (lane == 0 && it >= 0) sm.u.rep.terms[it] = fmax(sm.u.rep.terms[it], v);
      }
    }
    __syncwarp();
    // (3) terms exp(bm[r, j] - M_r), summed over the rows in ascending order
    for (int i0 = 0; i0 < n_items; i0 += 32) {
      const int item = i0 + lane;
      const double m_r = __shfl_sync(0xffffffffu, m_lane, item % nrows);
      if (item < n_items) {
        const double bmx = sm.u.rep.terms[item];
        sm.u.rep.terms[item] = (m_r == -INFINITY || bmx == -INFINITY) ? 0.0 : exp(bmx - m_r);
      }
    }
    __syncwarp();
    if (lane < n_rep) {
      double sum = 0.0;
      for (int rr = 0; rr < nrows; ++rr) sum += sm.u.rep.terms[lane * nrows + rr];
      sm.rep_val[lane] = sum;
    }
    __syncwarp();
    // re-sort the repaired runs by (exact score desc, block asc); a run never crosses the groups
    if (lane == 0) {
      int m0 = 0;
      while (m0 < n_rep) {
        int m1 = m0;
        while (m1 + 1 < n_rep && sm.rep_pos[m1 + 1] == sm.rep_pos[m1] + 1 && sm.rep_pos[m1 + 1] != nh) ++m1;
        for (int x = m0 + 1; x <= m1; ++x) {
          const double vx = sm.rep_val[x];
          const unsigned long long kx = sm.v.key[sm.rep_pos[x]];
          int y = x - 1;
          while (y >= m0) {
            const double vy = sm.rep_val[y];
            const unsigned long long ky = sm.v.key[sm.rep_pos[y]];
            const bool before = (vx > vy) || (vx == vy && key_block(kx) < key_block(ky));
            if (!before) break;
            sm.rep_val[y + 1] = vy;
            sm.v.key[sm.rep_pos[y + 1]] = ky;
            --y;
          }
          sm.rep_val[y + 1] = vx;
          sm.v.key[sm.rep_pos[y + 1]] = kx;
        }
        m0 = m1 + 1;
      }
    }
    __syncwarp();
  }
  for (int k = lane; k < a.mask_pitch; k += 32) out[k] = (k < K) ? key_block(sm.v.key[k]) : -1;
  if (lane == 0) a.mask_len[mrow] = K;
}

// The rows kap_select_warp_kernel deferred (list in a.defer), a block per row, grid-stride.
template <int HD, int KB>
__global__ void __launch_bounds__(kSelectThreads, 3) kap_select_kernel(KapArgs a, int cap) {
  const int n = a.defer[0];
  for (int li = blockIdx.x; li < n; li += gridDim.x) {
    kap_select_row<HD, KB>(a, cap, a.defer[1 + li]);
    __syncthreads();   // shared memory is reused by the next row
  }
}

template <typename T>
T* carve(uint8_t*& p, size_t n) {
  uintptr_t x = (reinterpret_cast<uintptr_t>(p) + 255) & ~uintptr_t(255);
  T* r = reinterpret_cast<T*>(x);
  p = reinterpret_cast<uint8_t*>(x + n * sizeof(T));
  return r;
}

struct WsLayout {
  size_t rows, scores, words, padded;  // padded: sampled rows of one head summed over requests, 128-padded
  size_t bms;                          // block maxima: Hq * kb * sum_b nqb_b (nqb_b + 1) / 2, bounded above
};

WsLayout ws_layout(int num_reqs, int num_q_heads, int block_size, int stride, int total_tokens, int max_seqlen) {
  WsLayout w;
  const size_t nqb_max = (max_seqlen + block_size - 1) / block_size;
  w.rows = static_cast<size_t>(num_q_heads) * (static_cast<size_t>(total_tokens) / stride + num_reqs);
  w.scores = static_cast<size_t>(num_q_heads) * nqb_max * (static_cast<size_t>(total_tokens) / block_size + num_reqs);
  w.words = (nqb_max + 31) / 32;
  w.padded = static_cast<size_t>(total_tokens) / stride + static_cast<size_t>(num_reqs) * (kRowTile + 1);
  // sum_b sum_{i < nqb_b} pitch(i) <= sum_b nqb_b ((nqb_b + 1) / 2 + 16) <= (T / b + B) (nqb_max / 2 + 17)
  w.bms = static_cast<size_t>(num_q_heads) * (block_size / stride) * (nqb_max / 2 + 17) *
          (static_cast<size_t>(total_tokens) / block_size + num_reqs);
  return w;
}

template <int HD, int KB>
cudaError_t launch_kap_t(KapArgs a, size_t qs_rows, size_t ks_rows, cudaStream_t stream) {
  kap_setup_kernel<<<1, 256, 0, stream>>>(a);
  {
    const int rpmax = (a.max_seqlen / a.stride + 1 + kRowTile - 1) / kRowTile * kRowTile;
    dim3 g((rpmax + 255) / 256, a.num_reqs * (a.num_q_heads + a.num_kv_heads));
    kap_gather_kernel<HD><<<g, 256, 0, stream>>>(a);
  }
  CUtensorMap qs_map, ks_map;
  {
    const cuuint64_t dims_q[2] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(qs_rows)};
    const cuuint64_t dims_k[2] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(ks_rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(HD) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kRowTile)};
    if (!encode_tiled_bf16(&qs_map, a.qs, 2, dims_q, strides, box)) return cudaErrorInvalidValue;
    if (!encode_tiled_bf16(&ks_map, a.ks, 2, dims_k, strides, box)) return cudaErrorInvalidValue;
  }
  const size_t tsm = sizeof(KapTileSmem<HD>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kap_logits_kernel<HD, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(tsm));
  if (e != cudaSuccess) return e;
  const unsigned tiles = static_cast<unsigned>(a.num_reqs) * a.num_q_heads * a.nrow_tiles_max;
  kap_logits_kernel<HD, KB><<<tiles, kLogitsThreads, tsm, stream>>>(qs_map, ks_map, a);
  {
    const size_t rows = static_cast<size_t>(a.num_q_heads) * (static_cast<size_t>(a.total_tokens) / a.stride + a.num_reqs);
    const unsigned blocks = static_cast<unsigned>((rows + 31) / 32);   // 8 warps of 4 rows
    kap_exact_kernel<HD><<<blocks, 256, 0, stream>>>(a);
    kap_rescan_kernel<HD, KB><<<512, 256, 0, stream>>>(a);
  }
  kap_block_scores_kernel<KB><<<dim3(a.nqb_max, a.num_q_heads, a.num_reqs), 128, 0, stream>>>(a);
  int cap = kSelectThreads;   // the sort works on at least one key per thread
  while (cap < a.nqb_max) cap <<= 1;
  const size_t ssm = select_smem_bytes(cap);
  e = cudaFuncSetAttribute(kap_select_kernel<HD, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ssm));
  if (e != cudaSuccess) return e;
  const long long nrows_mask = static_cast<long long>(a.num_reqs) * a.num_q_heads * a.nqb_max;
  kap_select_warp_kernel<HD, KB><<<static_cast<unsigned>((nrows_mask + kWarpSelWarps - 1) / kWarpSelWarps),
                                   kWarpSelWarps * 32, 0, stream>>>(a);
  kap_select_kernel<HD, KB><<<static_cast<unsigned>(nrows_mask < 1024 ? nrows_mask : 1024), kSelectThreads, ssm,
                              stream>>>(a, cap);
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
  add(sizeof(float) * w.rows);
  add(sizeof(float) * w.rows);
  add(sizeof(int64_t) * (w.rows + 1));
  add(sizeof(float) * w.rows);
  add(sizeof(int32_t) * w.rows);
  add(sizeof(double) * w.rows);
  add(sizeof(float) * w.rows);
  add(sizeof(int32_t) * w.rows);
  add(sizeof(uint32_t) * w.rows * w.words);
  add(sizeof(float) * w.scores);
  add(sizeof(float) * w.scores);
  add(sizeof(int64_t) * (num_reqs + 1));
  add(sizeof(int64_t) * (num_reqs + 1));
  add(sizeof(uint16_t) * static_cast<size_t>(num_q_heads) * w.padded * 128);
  add(sizeof(uint16_t) * static_cast<size_t>(num_kv_heads) * w.padded * 128);
  add(sizeof(uint32_t) * (static_cast<size_t>(num_kv_heads) * w.padded / 32 + 1));
  add(sizeof(int32_t) * (static_cast<size_t>(num_reqs) * num_q_heads * ((max_seqlen + block_size - 1) / block_size) + 1));
  add(sizeof(int64_t) * (num_reqs + 1));
  add(sizeof(float) * w.bms);
  return n + 256;
}

namespace {
// Driver calls that identify the current context, reached through the runtime's entry-point query
// (the library links no driver stub).
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};
const CtxFns& ctx_fns() {
  static CtxFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  return f;
}

// Identifier of the context current on this thread (unique for the life of the process), or 0 if
// there is none or it cannot be read.
unsigned long long current_ctx_id() {
  const CtxFns& f = ctx_fns();
  if (f.get_current == nullptr || f.get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (f.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}
}  // namespace

cudaError_t kap_static_scratch(void** ptr) {
  // Host code cannot use the array's name as a device address: look the address up with the
  // device current.  The array lives in the module loaded into a context, so the address is cached
  // per context (a context created after cudaDeviceReset, or another context made current through
  // the driver API, gets its own lookup).
  static std::mutex mu;
  static unsigned long long ids[kMaxStaticContexts] = {};
  static void* addr[kMaxStaticContexts] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = current_ctx_id();
  if (id != 0) {
    for (int s = 0; s < kMaxStaticContexts; ++s)
      if (ids[s] == id) {
        *ptr = addr[s];
        return cudaSuccess;
      }
  }
  // not cached: the lookup itself makes the device's primary context current if no context is
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, cosa_kap_static_scratch);
  if (e != cudaSuccess) return e;
  if (id == 0) id = current_ctx_id();
  if (id != 0) {
    int s = 0;
    while (s < kMaxStaticContexts && ids[s] != 0) ++s;
    if (s == kMaxStaticContexts) s = static_cast<int>(id % kMaxStaticContexts);   // table full: replace one
    ids[s] = id;
    addr[s] = p;
  }
  *ptr = p;
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
  a.ascending = (L.flags & COSA_FLAG_ASCENDING_ORDER) ? 1 : 0;
  a.top_p = (L.flags & COSA_FLAG_TOP_P) ? 1 : 0;
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
  a.v1 = carve<float>(p, w.rows);
  a.v2 = carve<float>(p, w.rows);
  a.amb = carve<int64_t>(p, w.rows + 1);
  a.qnorm = carve<float>(p, w.rows);
  a.c1 = carve<int32_t>(p, w.rows);
  a.M = carve<double>(p, w.rows);
  a.err = carve<float>(p, w.rows);
  a.rflags = carve<int32_t>(p, w.rows);
  a.hrm_bits = carve<uint32_t>(p, w.rows * w.words);
  a.score = carve<float>(p, w.scores);
  a.score_err = carve<float>(p, w.scores);
  a.qs_off = carve<int64_t>(p, L.num_reqs + 1);
  a.ks_off = carve<int64_t>(p, L.num_reqs + 1);
  a.qs = carve<uint16_t>(p, static_cast<size_t>(L.num_q_heads) * w.padded * 128);
  a.ks = carve<uint16_t>(p, static_cast<size_t>(L.num_kv_heads) * w.padded * 128);
  a.kvalid = carve<uint32_t>(p, static_cast<size_t>(L.num_kv_heads) * w.padded / 32 + 1);
  a.defer = carve<int32_t>(p, static_cast<size_t>(L.num_reqs) * L.num_q_heads * a.nqb_max + 1);
  a.bm_off = carve<int64_t>(p, L.num_reqs + 1);
  a.bm = carve<float>(p, w.bms);
  if (static_cast<size_t>(p - static_cast<uint8_t*>(L.workspace)) > L.workspace_bytes) return cudaErrorInvalidValue;
  const int kb = a.kb;
  const size_t qs_rows = static_cast<size_t>(L.num_q_heads) * w.padded;
  const size_t ks_rows = static_cast<size_t>(L.num_kv_heads) * w.padded;
  if (L.head_dim == 128) {
    if (kb == 8) return launch_kap_t<128, 8>(a, qs_rows, ks_rows, stream);
    if (kb == 4) return launch_kap_t<128, 4>(a, qs_rows, ks_rows, stream);
    if (kb == 16) return launch_kap_t<128, 16>(a, qs_rows, ks_rows, stream);
  } else if (L.head_dim == 64) {
    if (kb == 8) return launch_kap_t<64, 8>(a, qs_rows, ks_rows, stream);
    if (kb == 4) return launch_kap_t<64, 4>(a, qs_rows, ks_rows, stream);
    if (kb == 16) return launch_kap_t<64, 16>(a, qs_rows, ks_rows, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace cosa
