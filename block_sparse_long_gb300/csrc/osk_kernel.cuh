// Ordered-Skipping Kernel (OSK): block-sparse prefill attention over a paged KV cache.
//
// CoSA (arXiv 2607.25291), Sec. 4.3 and Algorithm A (ordered-skipping stage).  A persistent CTA per SM walks the
// work items with a grid stride; an item is a (request, query head, query block) with the 128-row
// tile of its query block (block_size 64 is padded to 128 rows), its ordered list of key blocks (the
// computation-order mask M_KAP) and the online-softmax state of its rows.
//
// Warp roles (384 threads):
//   warps 0-7  softmax, two warpgroups.  Thread (g, t) with g = warp / 4 and t the TMEM lane
//              (row) owns columns [g*b/2, (g+1)*b/2) of row t.  Per visit: read the row's half of
//              S = Q K^T from TMEM, apply the causal / length / missing-page masks, vote on the skip
//              (Eq. (5): skip iff every row has m_loc - m < ln(Delta/L)); for computed blocks combine
//              the halves' row maxima, update the running max and write P = exp(S - m_ref) as bf16
//              into TMEM for the P.V product.
//   warp 8     K producer: scans the mask row (drops invalid and repeated IDs, keeps the first
//              occurrence), resolves each kept block to physical pages through the page table
//              and TMA-gathers the K pages in mask order ("physical page jumping" and "any-order
//              page visiting" of Sec. 4.3).
//   warps 9/11 S issuers (warp 9 owns TMEM): S = Q K^T for the even / odd visits, each into its own
//              TMEM buffer, so two products are in flight while the softmax reads a third.
//   warp 10    V producer and O issuer: V pages only for blocks the vote computed, then
//              O += P V (P from TMEM, V from shared memory).
//
// The kernel is a template over the block, head and page sizes and three switches (binary-mask
// walk, skip rule on, visit flags recorded); each page size's instances are compiled in their own
// translation unit (osk_p16.cu ... osk_p128.cu).
//
// The running max m used by the skip rule is exact for the fp32 logits.  The reference
// max m_ref used for the exponentials lags it by up to 2^8 (rescaling O in TMEM only
// when m rises further), which changes rounding, not the result.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "cosa.h"
#include "internal.h"
#include "ptx.cuh"

namespace cosa {
namespace {

constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 256;
constexpr int kWarpK = 8, kWarpMma = 9, kWarpV = 10, kWarpS2 = 11;
constexpr int kMaxBlocksPerReq = 32768;  // dedupe bitmap capacity (blocks of one request)
constexpr int kMaxPagesPerBlock = 8;
constexpr float kRescaleLog2 = 8.0f;     // lazy-rescale threshold, log2 units
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO = 256, kTmemP0 = 384, kTmemP1 = 448;

struct alignas(16) KInfo {
  int32_t blk;     // block id, -1 = end of the list
  uint32_t pages;  // bit u set: page u of the block exists
  int32_t k;       // index of the entry in the mask row
  int32_t kvh;     // kv head of the work item
  int32_t phys[kMaxPagesPerBlock];
};

template <int BLK, int HD>
struct alignas(1024) OskSmem {
  static constexpr int NK = 3;
  static constexpr int NV = 2;
  static constexpr int TILE = BLK * HD * 2;   // bytes of one K or V tile
  static constexpr int HALF = BLK * 128;     // bytes of one 64-wide d chunk of a tile
  uint8_t q[128 * HD * 2];                    // [HD/64][128 rows][128 B], SW128
  uint8_t k[NK][TILE];                        // [HD/64][BLK rows][128 B], SW128
  uint8_t v[NV][TILE];
  uint64_t q_full, q_free;
  // k_full[slot][x]: K(v) landed, for the visits v of that slot with v % 2 == x.  A slot's visits
  // alternate between the two S issuers, and a parity wait only tells two phases apart: with one
  // barrier per slot, an issuer could wait for K(v) while K(v - NK) (the other issuer's) was still
  // in flight and take that earlier phase for its own.  Split by issuer, each barrier's phases are
  // waited for by one thread, in order.
  uint64_t k_full[NK][2], k_free[NK];
  uint64_t v_full[NV], v_free[NV];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[4];                         // per computed visit c: P written (slot c & 3)
  uint64_t o_done[2];
  uint64_t vreq_full[4];
  uint64_t cleanup;
  KInfo info[8];                              // visit info of visit v (slot v & 7), written with K(v)
  KInfo stage[32];                            // the K producer's current batch of 32 mask entries
  KInfo vreq[4];
  float pmax[2][2][128];                      // partial row maxima [visit & 1][column half][row]
  float lsum[2][128];                         // partial row sums, exchanged at the end
  int32_t pv_cmd[4];                          // per computed visit c: 2 = first of its item, 1 = accumulate, 0 = end
  uint32_t tmem_base;
  int32_t abort_flag;
  uint32_t seen[kMaxBlocksPerReq / 32];
};

struct OskArgs {
  const int32_t* cu_seqlens;
  const int32_t* page_table;
  const int32_t* mask;
  const int32_t* mask_len;
  uint16_t* out;
  uint8_t* visit_flags;
  int32_t* status;
  int num_reqs, num_q_heads, num_kv_heads, total_tokens, max_seqlen, nqb_max;
  int page_size, num_pages, max_pages_per_req, mask_pitch;
  int num_items;                      // kv heads * query blocks * requests * query heads per kv head
  int stall;                          // test hook: the K producer issues nothing (every wait runs out)
  float scale_log2;
  double skip_delta;
};

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// every page of the block exists and they occupy consecutive physical pages
template <typename Arr>
__device__ __forceinline__ bool pages_consecutive(uint32_t pages, uint32_t all_pages, const Arr& phys, int n) {
  if (pages != all_pages) return false;
  bool ok = true;
#pragma unroll
  for (int u = 1; u < kMaxPagesPerBlock; ++u)
    if (u < n) ok = ok && (phys[u] == phys[0] + u);
  return ok;
}

// Bounded wait taken by every lane of a warp; the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status) {
  return __all_sync(0xffffffffu, wait_parity_bounded(bar, parity, abort_flag, status));
}

template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 32) {
    tmem_st32(taddr, r);
  } else {
    static_assert(N == 16, "16 or 32 columns");
    tmem_st16(taddr, r);
  }
}

// Work item `idx` of the grid-stride order: kv-head major (a head's K/V stay in L2 while its
// query heads are processed), heaviest query blocks first.
struct Item {
  int b, h, kvh, i, tok0, L, nblk;
  int state;  // 0 run, 1 absent query block (shorter request), 2 bad cu_seqlens
};

__device__ __forceinline__ Item decode_item(const OskArgs& a, int idx, int blk) {
  Item it;
  const int G = a.num_q_heads / a.num_kv_heads;
  const int hg = idx % G;
  idx /= G;
  it.b = idx % a.num_reqs;
  idx /= a.num_reqs;
  it.i = a.nqb_max - 1 - (idx % a.nqb_max);
  it.kvh = idx / a.nqb_max;
  it.h = it.kvh * G + hg;
  it.tok0 = a.cu_seqlens[it.b];
  it.L = a.cu_seqlens[it.b + 1] - it.tok0;
  it.nblk = (it.L + blk - 1) / blk;
  if (it.L < 0 || it.L > a.max_seqlen || it.tok0 < 0 || it.tok0 + it.L > a.total_tokens) it.state = 2;
  else it.state = (it.i >= it.nblk) ? 1 : 0;
  return it;
}

// BIN: the mask rows are binary block masks walked in ascending order (logical skipping);
// SKIP: the in-kernel skip rule is on (Delta > 0); FLAGS: visit flags are recorded.  Fixing the
// last two, and the page size PSZ, at compile time keeps their tests out of the per-visit loops.
template <int BLK, int HD, int PSZ, bool BIN, bool SKIP, bool FLAGS>
__global__ void __launch_bounds__(kThreads, 1)
    osk_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap_blk,
               const __grid_constant__ CUtensorMap kmap_pg, const __grid_constant__ CUtensorMap vmap_blk,
               const __grid_constant__ CUtensorMap vmap_pg, const OskArgs a) {
  using S = OskSmem<BLK, HD>;
  constexpr int NK = S::NK, NV = S::NV;
  constexpr int DH = HD / 64;       // 64-wide d chunks
  constexpr int SC = BLK / 2;       // S columns per softmax thread
  constexpr int OC = HD / 2;        // O columns per softmax thread
  static_assert(NV * S::TILE >= 128 * HD * 2, "the V slots stage one output tile");
  extern __shared__ uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  constexpr int P = PSZ;
  constexpr int pages_per_blk = BLK / P;
  constexpr uint32_t all_pages = (1u << pages_per_blk) - 1u;
  static_assert(BLK % P == 0 && pages_per_blk <= kMaxPagesPerBlock, "a block is whole pages");
  volatile int* abort_flag = &sm.abort_flag;

  // ---------------- set-up (once per CTA) ----------------
  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_free, 2);        // one commit from each S issuer
    for (int s = 0; s < NK; ++s) {
      mbar_init(&sm.k_full[s][0], 1);
      mbar_init(&sm.k_full[s][1], 1);
      mbar_init(&sm.k_free[s], 1);
    }
    for (int s = 0; s < NV; ++s) { mbar_init(&sm.v_full[s], 1); mbar_init(&sm.v_free[s], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.s_full[s], 2);   // plain arrive (visit info) + UMMA commit
      mbar_init(&sm.s_free[s], 8);   // one per softmax warp
      mbar_init(&sm.o_done[s], 1);
    }
    for (int s = 0; s < 4; ++s) mbar_init(&sm.p_full[s], 8);
    for (int s = 0; s < 4; ++s) mbar_init(&sm.vreq_full[s], 1);
    mbar_init(&sm.cleanup, 3);       // one commit from each issuing warp
    sm.abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // padding rows 64..127 of a 64-row query block must hold finite values (their S rows are
  // discarded, but the UMMA reads them); Q loads never write them
  if (BLK < 128) {
    for (int e = threadIdx.x; e < DH * 64 * 8; e += kThreads) {
      const int dh = e / (64 * 8), rem = e % (64 * 8);
      reinterpret_cast<uint4*>(&sm.q[dh * 128 * 128 + 64 * 128])[rem] = make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  // Every role walks the same items (blockIdx.x, + gridDim.x, ...) and skips the same absent
  // or malformed ones.  Ring positions and barrier phases run on across items: v counts visits
  // (one extra per item for its end marker), c counts computed visits, n counts items.
  if (warp == kWarpK) {
    // =========================== K producer ===========================
    const uint32_t lane = lane_id();
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap_blk);
      tma_prefetch_desc(&kmap_pg);
      tma_prefetch_desc(&vmap_blk);
      tma_prefetch_desc(&vmap_pg);
    }
    int v = 0, n = 0;
    bool ok = !a.stall;
    for (int idx = blockIdx.x; idx < a.num_items && ok; idx += gridDim.x) {
      const Item it = decode_item(a, idx, BLK);
      if (it.state == 2 && lane == 0) report_status(a.status, kStatusBadInput);
      if (it.state != 0) continue;
      const int i = it.i, nblk = it.nblk, kvh = it.kvh;
      const int req_pages = (it.L + P - 1) / P;
      const size_t row_base = ((static_cast<size_t>(it.b) * a.num_q_heads + it.h) * a.nqb_max + i);
      const int32_t* mask_row = a.mask + row_base * a.mask_pitch;
      uint8_t* flags_row = FLAGS ? a.visit_flags + row_base * a.mask_pitch : nullptr;
      int n_entries = a.mask_len[row_base];
      n_entries = n_entries < 0 ? 0 : (n_entries > a.mask_pitch ? a.mask_pitch : n_entries);
      for (int w = lane; w < (nblk + 31) / 32; w += 32) sm.seen[w] = 0u;
      if (flags_row)
        for (int k = n_entries + lane; k < a.mask_pitch; k += 32) flags_row[k] = kVisitIgnored;
      __syncwarp();
      // Q of this item, once every Q K^T product of the previous item has completed
      if (n > 0) ok = warp_wait(&sm.q_free, (n - 1) & 1, abort_flag, a.status);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&sm.q_full, BLK * HD * 2);
        for (int dh = 0; dh < DH; ++dh)
          tma_load_4d(&sm.q[dh * 128 * 128], &qmap, &sm.q_full, 0, it.tok0 + i * BLK, dh, it.h);
      }
      ++n;
      const int32_t* pt_row = a.page_table + static_cast<size_t>(it.b) * a.max_pages_per_req;
      // binary mask: entry k selects block k; every causal block k < n_walk takes a turn through
      // the pipeline, the unselected ones as empty visits
      const int n_walk = BIN ? min(n_entries, i + 1) : 0;
      for (int k0 = 0; k0 < n_entries && ok; k0 += 32) {
        const int k = k0 + static_cast<int>(lane);
        const int j = (k < n_entries) ? (BIN ? (mask_row[k] != 0 ? k : -1) : mask_row[k]) : -1;
        const bool valid = (k < n_entries) && j >= 0 && j <= i && j < nblk;
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? j : -1 - static_cast<int>(lane));
        const bool first = valid && (static_cast<int>(lane) == __ffs(peers) - 1);
        const bool dup = first && ((sm.seen[j >> 5] >> (j & 31)) & 1u);
        const bool keep = first && !dup;
        __syncwarp();
        if (keep) atomicOr(&sm.seen[j >> 5], 1u << (j & 31));
        if (flags_row && k < n_entries && !keep) flags_row[k] = kVisitIgnored;
        // physical pages of this lane's block
        int phys[kMaxPagesPerBlock];
        uint32_t pages = 0;
#pragma unroll
        for (int u = 0; u < kMaxPagesPerBlock; ++u) {
          phys[u] = -1;
          if (keep && u < pages_per_blk) {
            const int lp = j * pages_per_blk + u;
            const int pp = (lp < req_pages) ? pt_row[lp] : -1;
            if (pp >= 0 && pp < a.num_pages) { phys[u] = pp; pages |= 1u << u; }
          }
        }
        // each lane stages its entry's visit record; lane 0 issues the visits from the stage
        const bool issue = keep || (BIN && k < n_walk);
        if (issue) {
          KInfo& st = sm.stage[lane];
          st.blk = (BIN && !keep) ? -2 : j;
          st.pages = pages;
          st.k = k;
          st.kvh = kvh;
#pragma unroll
          for (int u = 0; u < kMaxPagesPerBlock; ++u) st.phys[u] = phys[u];
        }
        __syncwarp();
        unsigned todo = __ballot_sync(0xffffffffu, issue);
        while (todo && ok) {
          const int src = __ffs(todo) - 1;
          todo &= todo - 1;
          const int slot = v % NK;
          if (v >= NK) ok = warp_wait(&sm.k_free[slot], ((v / NK) - 1) & 1, abort_flag, a.status);
          if (!ok) break;
          if (lane == 0) {
            const KInfo& st = sm.stage[src];
            KInfo& ki = sm.info[v & 7];
            ki = st;
            const int jj = st.blk;
            const uint32_t pg = st.pages;
            const int32_t* ph = st.phys;
            if (BIN && jj < 0) {
              // a block the binary mask drops: nothing to load
              mbar_arrive(&sm.k_full[slot][v & 1]);
            } else if (pages_consecutive(pg, all_pages, ph, pages_per_blk)) {
              // the block's pages follow each other in the cache: one copy of the whole tile
              mbar_arrive_expect_tx(&sm.k_full[slot][v & 1], BLK * HD * 2);
              tma_load_4d(&sm.k[slot][0], &kmap_blk, &sm.k_full[slot][v & 1], 0, ph[0] * P, 0, kvh);
            } else {
              const uint32_t bytes = static_cast<uint32_t>(__popc(pg)) * DH * P * 128u;
              mbar_arrive_expect_tx(&sm.k_full[slot][v & 1], bytes);
              for (int u = 0; u < pages_per_blk; ++u) {
                if (!((pg >> u) & 1u)) continue;
                for (int dh = 0; dh < DH; ++dh)
                  tma_load_4d(&sm.k[slot][dh * S::HALF + u * P * 128], &kmap_pg, &sm.k_full[slot][v & 1], 0, ph[u] * P, dh, kvh);
              }
            }
          }
          __syncwarp();
          ++v;
        }
      }
      // two end markers, one in each S issuer's half of the visit sequence
      for (int e2 = 0; e2 < 2 && ok; ++e2) {
        const int slot = v % NK;
        if (v >= NK) ok = warp_wait(&sm.k_free[slot], ((v / NK) - 1) & 1, abort_flag, a.status);
        if (ok && lane == 0) {
          sm.info[v & 7].blk = -1;
          mbar_arrive(&sm.k_full[slot][v & 1]);
        }
        __syncwarp();
        ++v;
      }
    }
    // on abort, let every issued copy land before the CTA exits
    if (*abort_flag && lane == 0) {
      if (n > 0) wait_parity_bounded(&sm.q_full, (n - 1) & 1, nullptr, nullptr);
      for (int s = 0; s < NK; ++s) {
        for (int x = 0; x < 2; ++x) {
          // visits u < v of slot s with u % 2 == x are u = r, r + 2 NK, ...
          const int r = (s % 2 == x) ? s : s + NK;
          const int issued = (v > r) ? (v - r + 2 * NK - 1) / (2 * NK) : 0;
          if (issued > 0) wait_parity_bounded(&sm.k_full[s][x], (issued - 1) & 1, nullptr, nullptr);
        }
      }
    }
  } else if (warp == kWarpMma || warp == kWarpS2) {
    // =========================== S issuers (lane 0 of two warps) ===========================
    // Issuer X takes the visits v with v % 2 == X and owns S buffer X: S(v) = Q K_v^T once K(v)
    // has landed and the softmax has read S(v - 2).  Two issuing threads keep two products in
    // flight (one thread issues a product's dependent steps one after another).
    if (lane_id() == 0) {
      const int X = (warp == kWarpMma) ? 0 : 1;
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, BLK, false, false);
      // descriptors differ from these bases only in the start-address field (address >> 4)
      const uint64_t qdesc = smem_desc_sw128(smem_u32(&sm.q[0]), 16, 1024);
      const uint64_t kdesc = smem_desc_sw128(smem_u32(&sm.k[0][0]), 16, 1024);
      int vv = X, n = 0;
      bool ok = true;
      for (int idx = blockIdx.x; idx < a.num_items && ok; idx += gridDim.x) {
        const Item it = decode_item(a, idx, BLK);
        if (it.state != 0) continue;
        ok = wait_parity_bounded(&sm.q_full, n & 1, abort_flag, a.status);
        ++n;
        tc_fence_after();
        while (ok) {
          const int slot = vv % NK, sb = X;
          if (!wait_parity_bounded(&sm.k_full[slot][X], (vv / (2 * NK)) & 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          if (vv >= 2 && !wait_parity_bounded(&sm.s_free[sb], ((vv >> 1) - 1) & 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          // info[vv & 7] is rewritten with K(vv + 8), long after the softmax has read it
          const int blk = sm.info[vv & 7].blk;
          mbar_arrive(&sm.s_full[sb]);
          if (blk < 0) {
            // end of the item (-1) or a dropped block (-2): no product; the K slot and the S
            // buffer pass on unused
            mbar_arrive(&sm.s_full[sb]);
            mbar_arrive(&sm.k_free[slot]);
            vv += 2;
            if (!BIN || blk == -1) break;
            continue;
          }
          tc_fence_after();
          const uint64_t kslot = kdesc + static_cast<uint64_t>(slot * (S::TILE >> 4));
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint64_t ad = qdesc + static_cast<uint64_t>(((kk >> 2) * 128 * 128 + (kk & 3) * 32) >> 4);
            const uint64_t bd = kslot + static_cast<uint64_t>(((kk >> 2) * S::HALF + (kk & 3) * 32) >> 4);
            umma_ss(tmem + (sb ? kTmemS1 : kTmemS0), ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
          }
          umma_commit(&sm.s_full[sb]);
          umma_commit(&sm.k_free[slot]);
          vv += 2;
        }
        // Q may be replaced once this item's products have completed
        if (ok) umma_commit(&sm.q_free);
      }
      // every issued UMMA finishes before TMEM is released
      umma_commit(&sm.cleanup);
      wait_parity_bounded(&sm.cleanup, 0, nullptr, nullptr);
    }
    __syncwarp();
  } else if (warp == kWarpV) {
    // =========================== V loads and O issue ===========================
    // For the c-th computed visit: load V_c as soon as the vote requests it, then O += P_c V_c once
    // P_c is in TMEM and V_c has landed (the first computed visit of an item overwrites O).  The
    // softmax requests V_{c+1} only after it has handed over P_c, so taking the two steps in this
    // order never waits on a later request.
    const uint32_t lane = lane_id();
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, HD, false, true);
    const uint64_t vdesc = smem_desc_sw128(smem_u32(&sm.v[0][0]), S::HALF, 1024);
    int c = 0;
    bool ok = true;
    while (ok) {
      if (!warp_wait(&sm.vreq_full[c & 3], (c >> 2) & 1, abort_flag, a.status)) { ok = false; break; }
      const KInfo r = sm.vreq[c & 3];
      if (r.blk < 0) break;
      const int slot = c % NV;
      if (c >= NV && !warp_wait(&sm.v_free[slot], ((c / NV) - 1) & 1, abort_flag, a.status)) {
        ok = false;
        break;
      }
      if (r.pages != all_pages) {
        // rows of pages that do not exist are zero: P is 0 there, and 0 * V must stay 0
        for (int u = 0; u < pages_per_blk; ++u) {
          if ((r.pages >> u) & 1u) continue;
          for (int dh = 0; dh < DH; ++dh) {
            uint4* z = reinterpret_cast<uint4*>(&sm.v[slot][dh * S::HALF + u * P * 128]);
            for (int e = lane; e < P * 8; e += 32) z[e] = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        if (pages_consecutive(r.pages, all_pages, r.phys, pages_per_blk)) {
          mbar_arrive_expect_tx(&sm.v_full[slot], BLK * HD * 2);
          tma_load_4d(&sm.v[slot][0], &vmap_blk, &sm.v_full[slot], 0, r.phys[0] * P, 0, r.kvh);
        } else {
          const uint32_t bytes = static_cast<uint32_t>(__popc(r.pages)) * DH * P * 128u;
          mbar_arrive_expect_tx(&sm.v_full[slot], bytes);
          for (int u = 0; u < pages_per_blk; ++u) {
            if (!((r.pages >> u) & 1u)) continue;
            for (int dh = 0; dh < DH; ++dh)
              tma_load_4d(&sm.v[slot][dh * S::HALF + u * P * 128], &vmap_pg, &sm.v_full[slot], 0, r.phys[u] * P, dh, r.kvh);
          }
        }
      }
      __syncwarp();
      if (!warp_wait(&sm.p_full[c & 3], (c >> 2) & 1, abort_flag, a.status)) { ok = false; break; }
      const int cmd = sm.pv_cmd[c & 3];
      if (!warp_wait(&sm.v_full[slot], (c / NV) & 1, abort_flag, a.status)) { ok = false; break; }
      if (lane == 0) {
        tc_fence_after();
        const uint32_t pcol = (c & 1) ? kTmemP1 : kTmemP0;
        const uint64_t vslot = vdesc + static_cast<uint64_t>(slot * (S::TILE >> 4));
#pragma unroll
        for (int kk = 0; kk < BLK / 16; ++kk) {
          const uint64_t bd = vslot + static_cast<uint64_t>((kk * 16 * 128) >> 4);
          umma_ts(tmem + kTmemO, tmem + pcol + kk * 8, bd, idesc_pv, (cmd == 1 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&sm.v_free[slot]);
        umma_commit(&sm.o_done[c & 1]);
      }
      __syncwarp();
      ++c;
    }
    if (lane == 0) {
      umma_commit(&sm.cleanup);
      wait_parity_bounded(&sm.cleanup, 0, nullptr, nullptr);
      if (*abort_flag) {
        for (int s2 = 0; s2 < NV; ++s2) {
          const int issued = (c - s2 + NV - 1) / NV;
          if (issued > 0) wait_parity_bounded(&sm.v_full[s2], (issued - 1) & 1, nullptr, nullptr);
        }
      }
    }
    __syncwarp();
  } else {
    // =========================== softmax warpgroups (warps 0-7) ===========================
    const int g = warp >> 2;              // column half
    const int t = (warp & 3) * 32 + static_cast<int>(lane_id());   // tile row == TMEM lane
    const uint32_t lane = lane_id();
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int col0 = g * SC;              // first S column of this thread
    constexpr bool use_skip = SKIP;
    const float sl2 = a.scale_log2;
    constexpr int pshift = (P == 16) ? 4 : (P == 32) ? 5 : (P == 64) ? 6 : 7;
    const bool leader = threadIdx.x == 0;
    int v = 0;                 // visits, all items
    int c = 0;                 // computed visits, all items
    bool ok = true;
    bool local_fail = false;   // a wait of this warp ran out after the last vote
    for (int idx = blockIdx.x; idx < a.num_items && ok; idx += gridDim.x) {
      const Item it = decode_item(a, idx, BLK);
      if (it.state != 0) continue;
      const int i = it.i, L = it.L;
      const int pos = i * BLK + t;          // token position of this row inside the request
      const bool row_valid = (t < BLK) && (pos < L);
      // ln(Delta / L) in log2 units, in fp32 (the logits it is compared with are fp32)
      const float tau2 = use_skip ? log2f(static_cast<float>(a.skip_delta)) - log2f(static_cast<float>(L)) : 0.0f;
      const size_t row_base = ((static_cast<size_t>(it.b) * a.num_q_heads + it.h) * a.nqb_max + i);
      uint8_t* flags_row = FLAGS ? a.visit_flags + row_base * a.mask_pitch : nullptr;
      float m_run = -INFINITY;   // running max (log2 units), Algorithm A (running-max update)
      float m_ref = -INFINITY;   // max the exponentials are taken against
      float l_part = 0.0f;       // this half's share of the row sum l
      int c_item = 0;            // computed visits of this item
      for (;; ++v) {
        const int sb = v & 1;
        const uint32_t sbase = tmem + lane_addr + (sb ? kTmemS1 : kTmemS0) + col0;
        int ki_blk = -1, ki_k = 0;
        uint32_t ki_pages = 0;
        float sv[SC];
        float pm = -INFINITY;   // this half's row max of the block (raw logits)
        bool okw = !local_fail && wait_parity_bounded(&sm.s_full[sb], (v >> 1) & 1, abort_flag, a.status);
        okw = __all_sync(0xffffffffu, okw);
        if (okw) {
          // slot v & 7 is rewritten with K(v + 8), which waits for S(v + 3) to be released
          const int4 hd = *reinterpret_cast<const int4*>(&sm.info[v & 7]);
          ki_blk = hd.x;
          ki_pages = static_cast<uint32_t>(hd.y);
          ki_k = hd.z;
          if (ki_blk >= 0) {
            // the load also reduces: pm = max of this thread's columns of S, before any mask
            tc_fence_after();
            if constexpr (SC == 64) {
              uint32_t r[64];
              tmem_ld64_max(sbase, r, pm);
              tmem_wait_ld();
              reg_after_wait(pm);
#pragma unroll
              for (int e = 0; e < 64; ++e) sv[e] = __uint_as_float(r[e]);
            } else {
              static_assert(SC == 32, "32 or 64 S columns per thread");
              uint32_t r[32];
              tmem_ld32_max(sbase, r, pm);
              tmem_wait_ld();
              reg_after_wait(pm);
#pragma unroll
              for (int e = 0; e < 32; ++e) sv[e] = __uint_as_float(r[e]);
            }
            tc_fence_before();
          }
          // the buffer is released for every visit, the end marker's included
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.s_free[sb]);
          if (ki_blk >= 0) {
            // masks: causal on the diagonal block, length on the last block, missing pages
            const int key0 = ki_blk * BLK;
            const bool need_mask = (ki_blk == i) || (key0 + BLK > L) || (ki_pages != all_pages) || !row_valid;
            if (need_mask) {
              // masked columns leave the maximum: take it again over the masked values
              const int lim = row_valid ? min(pos, L - 1) - key0 : -1;  // last visible column
#pragma unroll
              for (int e = 0; e < SC; ++e)
                if (col0 + e > lim || !((ki_pages >> ((col0 + e) >> pshift)) & 1u)) sv[e] = -INFINITY;
              static_assert(SC % 16 == 0, "16-column groups");
              float m4[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) m4[q] = sv[q];
#pragma unroll
              for (int e = 4; e < SC; e += 4) {
#pragma unroll
                for (int q = 0; q < 4; ++q) m4[q] = fmaxf(m4[q], sv[e + q]);
              }
              pm = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            }
          }
        }
        // skip vote (Eq. (5)).  A row wants the block iff m_loc - max(m_run, m_loc) >= tau2; that
        // test is monotone in m_loc, so it holds for the row iff it holds for one of the two
        // column halves' partial maxima, and the block is computed iff some half of some row wants it.
        const float p_loc = (pm == -INFINITY) ? -INFINITY : pm * sl2;
        bool want = true;
        if (use_skip) want = row_valid && (p_loc != -INFINITY) && (p_loc - fmaxf(m_run, p_loc) >= tau2);
        // The partial row maxima go to shared memory before the vote (double-buffered by visit) and
        // are read after it.  First barrier: some row wants the block, or the visit ends the item,
        // or a wait ran out (all warps whose waits succeed see the same visit record); only then
        // a second barrier tells these apart, so a skipped block costs one barrier.
        sm.pmax[v & 1][g][t] = pm;
        const bool stop = !okw || (ki_blk < 0);
        bool compute = named_bar_red_or(2, kSoftmaxThreads, want || stop);
        if (compute && named_bar_red_or(1, kSoftmaxThreads, stop)) {
          if (named_bar_red_or(2, kSoftmaxThreads, !okw)) ok = false;
          if (BIN && ok && ki_blk == -2) continue;   // a block the binary mask drops
          if (ok) {
            // the item's second end marker (the other S issuer's): release that buffer too
            const int v1 = v + 1;
            bool ok2 = wait_parity_bounded(&sm.s_full[v1 & 1], (v1 >> 1) & 1, abort_flag, a.status);
            ok2 = __all_sync(0xffffffffu, ok2);
            if (ok2) {
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.s_free[v1 & 1]);
            } else {
              ok = false;
            }
          }
          v += 2;
          break;
        }
        // a skipped block leaves every row's running max unchanged (m_loc < m_run + tau2 <= m_run)
        float m_new = m_run;
        if (compute) {
          const float mx = fmaxf(sm.pmax[v & 1][0][t], sm.pmax[v & 1][1][t]);
          const float m_loc = (mx == -INFINITY) ? -INFINITY : mx * sl2;
          m_new = fmaxf(m_run, m_loc);
        }
        m_run = m_new;
        if (leader && flags_row) flags_row[ki_k] = compute ? kVisitComputed : kVisitSkipped;
        if (!compute) continue;
        if (leader) {
          sm.pv_cmd[c & 3] = (c_item == 0) ? 2 : 1;
          sm.vreq[c & 3] = sm.info[v & 7];
          mbar_arrive(&sm.vreq_full[c & 3]);
        }
        // lazy rescale of O and l when the max rises by more than 2^8
        const bool first_mass = (m_ref == -INFINITY) && (m_new != -INFINITY);
        const bool rescale = (m_ref != -INFINITY) && (m_new > m_ref + kRescaleLog2);
        float alpha = 1.0f;
        if (first_mass) m_ref = m_new;
        if (rescale) {
          alpha = ex2_approx(m_ref - m_new);
          m_ref = m_new;
          l_part *= alpha;
        }
        // P = exp2(S * scale * log2(e) - m_ref) as bf16 pairs; masked entries are -inf -> 0
        const float base = (m_ref == -INFINITY) ? 0.0f : m_ref;
        uint32_t pk[SC / 2];
        float rs4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int e = 0; e < SC / 2; ++e) {
          float x0, x1;
          fma2_bc(x0, x1, sv[2 * e], sv[2 * e + 1], sl2, -base);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          add2_acc(rs4[(e & 1) * 2], rs4[(e & 1) * 2 + 1], p0, p1);
          pk[e] = pack_bf16x2(p0, p1);
        }
        l_part += (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        // the P buffer written now was read by the P.V two computed visits ago
        if (c >= 2) {
          bool okp = wait_parity_bounded(&sm.o_done[c & 1], ((c - 2) >> 1) & 1, abort_flag, a.status);
          if (!__all_sync(0xffffffffu, okp)) { local_fail = true; continue; }
        }
        tc_fence_after();
        tmem_st_n<SC / 2>(tmem + lane_addr + ((c & 1) ? kTmemP1 : kTmemP0) + g * (SC / 2), pk);
        tmem_wait_st();
        // O (this half's columns) is scaled once every earlier P.V of the item has landed; P.V of
        // this visit is issued only after p_full, so it accumulates onto the scaled O
        if (__any_sync(0xffffffffu, rescale) && c_item > 0) {
          bool okr = wait_parity_bounded(&sm.o_done[(c - 1) & 1], ((c - 1) >> 1) & 1, abort_flag, a.status);
          if (!__all_sync(0xffffffffu, okr)) { local_fail = true; continue; }
          tc_fence_after();
          const uint32_t ob = tmem + lane_addr + kTmemO + g * OC;
#pragma unroll 1
          for (int cc = 0; cc < OC / 16; ++cc) {
            uint32_t r[16];
            tmem_ld16(ob + cc * 16, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st16(ob + cc * 16, r);
            tmem_wait_st();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[c & 3]);
        ++c;
        ++c_item;
      }
      if (!ok) break;
      // ---------------- epilogue: O / l -> bf16 -> global ----------------
      if (c_item > 0) ok = wait_parity_bounded(&sm.o_done[(c - 1) & 1], ((c - 1) >> 1) & 1, abort_flag, a.status);
      ok = named_bar_red_or(1, kSoftmaxThreads, !ok) ? false : ok;
      if (!ok) break;
      tc_fence_after();
      sm.lsum[g][t] = l_part;
      named_bar_sync(3, kSoftmaxThreads);
      const float l_sum = sm.lsum[0][t] + sm.lsum[1][t];
      const float inv_l = (l_sum > 0.0f) ? 1.0f / l_sum : 0.0f;
      // the V slots are idle here: this item's P.V products are done, the next item's V loads
      // follow its first vote
      uint8_t* stage = &sm.v[0][0];
      constexpr int CH = HD / 8;  // 16-byte chunks per output row
      {
        const uint32_t ob = tmem + lane_addr + kTmemO + g * OC;
#pragma unroll
        for (int cc = 0; cc < OC / 32; ++cc) {
          uint32_t r[32];
          if (c_item > 0) {
            tmem_ld32(ob + cc * 32, r);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = 0u;
          }
          // 32 fp32 -> 16 packed bf16 pairs -> four 16-byte chunks, XOR-swizzled by row
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[q4 * 8 + 0]) * inv_l, __uint_as_float(r[q4 * 8 + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(r[q4 * 8 + 2]) * inv_l, __uint_as_float(r[q4 * 8 + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(r[q4 * 8 + 4]) * inv_l, __uint_as_float(r[q4 * 8 + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(r[q4 * 8 + 6]) * inv_l, __uint_as_float(r[q4 * 8 + 7]) * inv_l);
            const int chunk = (g * OC) / 8 + cc * 4 + q4;   // 16-byte chunk of the row
            const int phys_chunk = chunk ^ (t & (CH - 1));
            *reinterpret_cast<uint4*>(stage + t * (HD * 2) + phys_chunk * 16) = w;
          }
        }
      }
      tc_fence_before();
      named_bar_sync(3, kSoftmaxThreads);
      {
        const int rows = min(BLK, L - i * BLK);
        uint8_t* out = reinterpret_cast<uint8_t*>(a.out);
        const int tid = g * 128 + t;
        for (int e = tid; e < rows * CH; e += kSoftmaxThreads) {
          const int r = e / CH, chunk = e % CH;
          const uint4 w = *reinterpret_cast<const uint4*>(stage + r * (HD * 2) + ((chunk ^ (r & (CH - 1))) * 16));
          const size_t tok = static_cast<size_t>(it.tok0) + static_cast<size_t>(i) * BLK + r;
          *reinterpret_cast<uint4*>(out + ((tok * a.num_q_heads + it.h) * HD) * 2 + chunk * 16) = w;
        }
      }
      // the staging reads finish before a later TMA load may refill the V slots
      fence_proxy_async_smem();
      named_bar_sync(3, kSoftmaxThreads);
    }
    // end markers for the V producer and the O issuer
    if (leader) {
      sm.vreq[c & 3].blk = -1;
      mbar_arrive(&sm.vreq_full[c & 3]);
      sm.pv_cmd[c & 3] = 0;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.p_full[c & 3]);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int BLK, int HD, int PSZ, bool BIN, bool SKIP, bool FLAGS>
cudaError_t launch_osk_b(const OskLaunch& L, cudaStream_t stream) {
  OskArgs a;
  a.cu_seqlens = L.cu_seqlens;
  a.page_table = L.page_table;
  a.mask = L.mask;
  a.mask_len = L.mask_len;
  a.out = reinterpret_cast<uint16_t*>(L.out);
  a.visit_flags = L.visit_flags;
  a.status = L.status;
  a.num_reqs = L.num_reqs;
  a.num_q_heads = L.num_q_heads;
  a.num_kv_heads = L.num_kv_heads;
  a.total_tokens = L.total_tokens;
  a.max_seqlen = L.max_seqlen;
  a.nqb_max = (L.max_seqlen + BLK - 1) / BLK;
  a.page_size = L.page_size;
  a.num_pages = L.num_pages;
  a.max_pages_per_req = L.max_pages_per_req;
  a.mask_pitch = L.mask_pitch;
  a.scale_log2 = static_cast<float>(L.sm_scale * 1.4426950408889634);
  a.skip_delta = L.skip_delta;
  a.stall = (L.flags & COSA_FLAG_TEST_STALL) ? 1 : 0;
  const size_t smem = sizeof(OskSmem<BLK, HD>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(osk_kernel<BLK, HD, PSZ, BIN, SKIP, FLAGS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long items =
      static_cast<long long>(L.num_kv_heads) * a.nqb_max * L.num_reqs * (L.num_q_heads / L.num_kv_heads);
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.num_items = static_cast<int>(items);
  // persistent: one CTA per SM walks the items with a grid stride
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
  osk_kernel<BLK, HD, PSZ, BIN, SKIP, FLAGS><<<grid, kThreads, smem, stream>>>(L.qmap, L.kmap_blk, L.kmap_pg, L.vmap_blk, L.vmap_pg, a);
  return cudaGetLastError();
}

template <int BLK, int HD, int PSZ, bool BIN>
cudaError_t launch_osk_s(const OskLaunch& L, cudaStream_t stream) {
  const bool skip = L.skip_delta > 0.0, flags = L.visit_flags != nullptr;
  if (skip)
    return flags ? launch_osk_b<BLK, HD, PSZ, BIN, true, true>(L, stream)
                 : launch_osk_b<BLK, HD, PSZ, BIN, true, false>(L, stream);
  return flags ? launch_osk_b<BLK, HD, PSZ, BIN, false, true>(L, stream)
               : launch_osk_b<BLK, HD, PSZ, BIN, false, false>(L, stream);
}

// every instance of page size PSZ for the block and head sizes of the call
template <int PSZ>
cudaError_t launch_osk_page(const OskLaunch& L, cudaStream_t stream) {
  const bool bin = (L.flags & COSA_FLAG_BINARY_MASK) != 0;
  if (L.block_size == 128 && L.head_dim == 128)
    return bin ? launch_osk_s<128, 128, PSZ, true>(L, stream) : launch_osk_s<128, 128, PSZ, false>(L, stream);
  if (L.block_size == 128 && L.head_dim == 64)
    return bin ? launch_osk_s<128, 64, PSZ, true>(L, stream) : launch_osk_s<128, 64, PSZ, false>(L, stream);
  if constexpr (PSZ <= 64) {
    if (L.block_size == 64 && L.head_dim == 128)
      return bin ? launch_osk_s<64, 128, PSZ, true>(L, stream) : launch_osk_s<64, 128, PSZ, false>(L, stream);
    if (L.block_size == 64 && L.head_dim == 64)
      return bin ? launch_osk_s<64, 64, PSZ, true>(L, stream) : launch_osk_s<64, 64, PSZ, false>(L, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

// the instances of each page size, one translation unit each
cudaError_t launch_osk_p16(const OskLaunch& L, cudaStream_t stream);
cudaError_t launch_osk_p32(const OskLaunch& L, cudaStream_t stream);
cudaError_t launch_osk_p64(const OskLaunch& L, cudaStream_t stream);
cudaError_t launch_osk_p128(const OskLaunch& L, cudaStream_t stream);

}  // namespace cosa
