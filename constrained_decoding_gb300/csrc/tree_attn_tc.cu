// Tree attention on the 5th-generation tensor cores (head dim 128).
//
// Same queries, keys and visibility as the warp-MMA tree attention: prefix
// queries causal over the prefix, branch queries over the whole prefix plus
// their own ancestors (the per-field branch mask of parallel constrained
// decoding).  A CTA owns 128 query rows (whole tokens of one GQA group) and
// walks 64-key blocks:
//   S = Q K^T            tcgen05.mma, Q and K from shared memory, S in TMEM
//   P = exp2(S - m)      one thread per row reads its S row from TMEM
//   O += P V             tcgen05.mma, P (fp16) from TMEM, V as an
//                        MN-major operand, O accumulated in TMEM
// The running maximum m is only moved (and O, l rescaled) when a block's
// maximum exceeds it by more than 14 (log2 units): every P stays <= 2^14, a
// finite fp16, and the result is exact up to rounding, while the rescale
// (which waits for the previous P V) is rare.  Warp 0 loads K/V (TMA for
// prefix blocks, gathered cp.async for ancestor chunks), warp 1 issues the S
// MMAs and warp 6 the P V MMAs, warps 2-5 run the softmax and the epilogue;
// P goes back into TMEM over its own S columns and is the A operand of the
// P V MMA.  With fp16 rounding remainders, S takes Q K_lo + Q_lo K and O
// takes P V_lo + P_lo V (each set optional: a template variant per set).  A
// (csk, 1, 1) cluster splits a tile's key blocks and combines the partial
// softmax states through distributed shared memory.
#include <algorithm>
#include <climits>
#include <cstdint>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"
#include "ptx.cuh"
#include "warp_mma.cuh"

namespace pcd {
namespace {

constexpr int kRows = 128;                   // query rows per CTA (MMA M)
constexpr int kDH = 128;
constexpr int kKeys = 64;                    // keys per block
constexpr int kQBytes = kRows * kDH * 2;     // two 64-column halves of 16 KB
constexpr int kKVBytes = kKeys * kDH * 2;    // two 64-column halves of 8 KB
constexpr int kOffQ = 0;
constexpr int kOutLd = kDH * 2 + 16;         // staged output row (bytes): padded against bank conflicts
constexpr int kRedLd = kDH + 4;              // fp32 partial-O row stride for the cluster combine
constexpr uint32_t kColS = 0;

// Shared and tensor memory layout.  QLO: q and k also carry their fp16
// rounding remainders (a second tile next to each) for the S cross terms;
// VLO: v and P carry theirs for the P V cross terms.  Stages: 2 with both
// sets of remainders, 3 with one, 4 without any.
template <bool QLO, bool VLO>
struct TcCfg {
  static constexpr int kStages = (QLO && VLO) ? 2 : (QLO || VLO) ? 3 : 4;  // K and V stages: loads run ahead
  static constexpr int kQAll = kQBytes * (QLO ? 2 : 1);     // Q (then Q's remainder)
  static constexpr int kKSt = kKVBytes * (QLO ? 2 : 1);     // one K stage: hi, then lo
  static constexpr int kVSt = kKVBytes * (VLO ? 2 : 1);     // one V stage: hi, then lo
  static constexpr int kOffK = kQAll;
  static constexpr int kOffV = kOffK + kStages * kKSt;
  static constexpr int kOffBar = kOffV + kStages * kVSt;
  static constexpr int kOffML = kOffBar + 256;
  static constexpr int kSmem = kOffML + 2048 + 1024;      // + alignment slack
  // S (then P: hi in the first 32 columns, lo in the next 32) per stage, then O
  static constexpr uint32_t kColO = kStages * kKeys;
  static constexpr uint32_t kTmemCols = kColO + kDH <= 256 ? 256 : 512;
  static_assert(kColO + kDH <= kTmemCols, "S stages and O fit the TMEM allocation");
  static_assert(2 * kRows * kOutLd <= kOffBar, "staged hi and lo output rows fit the Q/K/V region");
  static_assert((kRows + 8) * kRedLd * 4 <= kOffBar, "received partial rows fit the Q/K/V region");
  static_assert((kRows + 8) * 8 <= 2048, "received (m, l) pairs fit their region");
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};
constexpr float kRescale = 14.f;             // log2 headroom before m moves: P <= 2^14 stays finite in fp16

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // 128-byte swizzled row of 8 16-byte chunks
  return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

template <bool QLO, bool VLO>
__global__ void __launch_bounds__(224, 1)
    tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmKlo, const __grid_constant__ CUtensorMap tmVlo,
                        const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQlo,
                        const TreeAttnArgs a, int layer, uint64_t wait_ns, int* err) {
  using C = TcCfg<QLO, VLO>;
  constexpr int kStages = C::kStages, kKSt = C::kKSt, kVSt = C::kVSt, kOffK = C::kOffK, kOffV = C::kOffV,
                kOffBar = C::kOffBar;
  constexpr int kOffML = C::kOffML;
  constexpr uint32_t kColO = C::kColO, kTmemCols = C::kTmemCols;
  extern __shared__ uint8_t tta_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tta_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* k_full = bars;        // [kStages] producer -> MMA
  uint64_t* v_full = bars + 4;    // [kStages]
  uint64_t* k_free = bars + 8;    // [kStages] MMA: the S that read the K stage is done -> producer
  uint64_t* v_free = bars + 12;   // [kStages] MMA: the P V that read the V stage is done -> producer
  uint64_t* s_full = bars + 16;   // [kStages] MMA: S ready -> softmax
  uint64_t* p_full = bars + 20;   // [kStages] softmax: P in TMEM -> MMA
  uint64_t* pv_done = bars + 24;  // [kStages] MMA: O += P V done (S/P columns free, O current)
  uint64_t* drain = bars + 28;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 29);
  uint64_t* q_full = bars + 30;   // producer: the Q tile (and remainder) landed -> MMA
  uint64_t* drain2 = bars + 31;   // the P V issuer's MMAs are done
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float2* sML = reinterpret_cast<float2*>(smem + kOffML);
  float* sRed = reinterpret_cast<float*>(smem);  // received partial rows, after the key loop

  const int csk = a.csk;
  const int item = blockIdx.x / csk;
  const int rank = blockIdx.x - item * csk;
  const int hk = blockIdx.y;
  const int G = a.Hq / a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const bool branch = item < a.n_br_tiles;
  const int tile = branch ? item : a.n_pf_tiles - 1 - (item - a.n_br_tiles);
  // a branch tile's tokens come from the plan (tiles end at request boundaries)
  const int t0 = branch ? a.tile_tok[3 * tile] : tile * a.tpt;
  const int ntok = branch ? a.tile_tok[3 * tile + 1] : min(a.tpt, a.n_pf - t0);
  const int qrow0 = branch ? a.br_row0 + t0 : t0;
  const int rows = ntok * G;
  // a batch's branch tile reads its own request's prefix cache
  const SegKV* sgk = (branch && a.segs) ? a.segs + a.tile_tok[3 * tile + 2] : nullptr;
  const int n_keys = sgk ? sgk->n_keys : a.n_keys;
  const int pf_keys = branch ? n_keys : min(n_keys, a.pf_pos0 + t0 + ntok);
  const int nbp = (pf_keys + kKeys - 1) / kKeys;
  const int ch0 = branch ? a.tile_chunk_off[tile] : 0;
  const int nb = nbp + (branch ? a.tile_chunk_off[tile + 1] - ch0 : 0);
  const int my_n = rank < nb ? (nb - 1 - rank) / csk + 1 : 0;
  // CTAs of one KV head start at different key blocks (the online softmax
  // takes them in any order), so they do not all read the same block at once
  const int rot = my_n > 0 ? static_cast<int>((item * 5u + hk * 3u) % static_cast<unsigned>(my_n)) : 0;
  auto block_of = [&](int i) { int j = i + rot; j -= j >= my_n ? my_n : 0; return rank + j * csk; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_free[s], 1);
      mbar_init(&v_free[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 128);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(drain, 1);
    mbar_init(drain2, 1);
    mbar_init(q_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    if constexpr (QLO) {
      tma_prefetch_desc(&tmQlo);
      tma_prefetch_desc(&tmKlo);
    }
    if constexpr (VLO) tma_prefetch_desc(&tmVlo);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  griddep_launch_dependents();
  griddep_wait();  // q, K and V come from the projection that ran just before

  auto fail = [&](int code) {
    record_error(err, code);
    *abort_flag = 1;
  };
  const int r = 32 * (warp & 3) + lane;  // query row (TMEM lane) of a softmax thread (warps 2-5)
  int kissued[kStages] = {}, vissued[kStages] = {};  // loads per K / V stage (producer warp)
  float m_ref = -INFINITY, l = 0.f;              // softmax state of row r
  bool have_o = false;

  if (warp == 0) {
    // ------------------------------------------------------------ K/V loads
    const act_t* kbp = a.kb + static_cast<size_t>(hk) * a.n_br * kDH;
    const act_t* vbp = a.vb + static_cast<size_t>(hk) * a.n_br * kDH;
    // this (layer, KV head)'s rows in a batch request's cache
    const size_t seg_off = sgk ? (static_cast<size_t>(a.layer) * a.Hkv + hk) * static_cast<size_t>(sgk->cap) * kDH : 0;
    const act_t* kblp = QLO ? a.kb_lo + static_cast<size_t>(hk) * a.n_br * kDH : nullptr;
    const act_t* vblp = VLO ? a.vb_lo + static_cast<size_t>(hk) * a.n_br * kDH : nullptr;
    // rows of K or V (and remainder) by cp.async: an ancestor chunk's rows of
    // the branch K/V by index (keys), or a batch request's prefix rows j0.. of
    // its own cache; zero past the end
    auto gather = [&](uint8_t* dst, const act_t* src, const act_t* src_lo, const int32_t* keys, int j0, int n_valid,
                      uint64_t* bar) {
      for (int e = lane; e < kKeys * 16; e += 32) {
        const int kr = e >> 4, c = e & 15;
        const int j = keys ? keys[kr] : j0 + kr;
        const bool ok = keys ? (j >= 0 && j < a.n_br) : j < n_valid;
        const size_t off = static_cast<size_t>(ok ? j : 0) * kDH + c * 8;
        const uint32_t so = (c >> 3) * (kKVBytes / 2) + swz(kr, c & 7);
        cp_async16(dst + so, src + off, ok);
        if (src_lo) cp_async16(dst + kKVBytes + so, src_lo + off, ok);
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
    };
    // a prefix block by TMA: both 64-column halves, and the remainder's (lo)
    auto tma_block = [&](uint8_t* dst, const CUtensorMap* hi, const CUtensorMap* lo, int b, uint64_t* bar) {
      mbar_arrive_expect_tx(bar, lo ? 2u * kKVBytes : static_cast<uint32_t>(kKVBytes));
      tma_load_4d(dst, hi, bar, 0, b * kKeys, hk, layer);
      tma_load_4d(dst + kKVBytes / 2, hi, bar, 64, b * kKeys, hk, layer);
      if (lo) {
        tma_load_4d(dst + kKVBytes, lo, bar, 0, b * kKeys, hk, layer);
        tma_load_4d(dst + kKVBytes + kKVBytes / 2, lo, bar, 64, b * kKeys, hk, layer);
      }
    };
    if (lane == 0) {
      // the Q tile: tpt tokens x G heads of this KV head, both 64-column
      // halves (and the remainder's), one box each; rows past tpt x G are
      // zeroed by the softmax warps
      const uint32_t box = 64u * static_cast<uint32_t>(G * a.tpt) * 2u;
      mbar_arrive_expect_tx(q_full, (QLO ? 4u : 2u) * box);
      tma_load_3d(smem + kOffQ, &tmQ, q_full, 0, hk * G, qrow0);
      tma_load_3d(smem + kOffQ + kQBytes / 2, &tmQ, q_full, 64, hk * G, qrow0);
      if constexpr (QLO) {
        tma_load_3d(smem + kOffQ + kQBytes, &tmQlo, q_full, 0, hk * G, qrow0);
        tma_load_3d(smem + kOffQ + kQBytes + kQBytes / 2, &tmQlo, q_full, 64, hk * G, qrow0);
      }
    }
    __syncwarp();
    for (int i = 0; i < my_n; ++i) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int s = i % kStages, b = block_of(i);
      const uint32_t fpar = static_cast<uint32_t>(((i - kStages) / kStages) & 1);  // phase of block i - kStages
      const int32_t* keys = b >= nbp ? a.tile_keys + static_cast<size_t>(ch0 + b - nbp) * kKeys : nullptr;
      // the K stage is free once the S of block i - kStages is computed
      if (!__all_sync(0xffffffffu, i < kStages || mbar_wait(&k_free[s], fpar, wait_ns))) {
        if (lane == 0) fail(DEV_WAIT_TIMEOUT_PRODUCER);
        break;
      }
      uint8_t* kd = smem + kOffK + s * kKSt;
      if (keys) {
        gather(kd, kbp, kblp, keys, 0, 0, &k_full[s]);
      } else if (sgk) {
        gather(kd, sgk->k + seg_off, QLO ? sgk->k_lo + seg_off : nullptr, nullptr, b * kKeys, pf_keys, &k_full[s]);
      } else {
        if (lane == 0) tma_block(kd, &tmK, QLO ? &tmKlo : nullptr, b, &k_full[s]);
      }
      ++kissued[s];
      // the V stage is free once the P V of block i - kStages is done
      if (!__all_sync(0xffffffffu, i < kStages || mbar_wait(&v_free[s], fpar, wait_ns))) {
        if (lane == 0) fail(DEV_WAIT_TIMEOUT_PRODUCER);
        break;
      }
      uint8_t* vd = smem + kOffV + s * kVSt;
      if (keys) {
        gather(vd, vbp, vblp, keys, 0, 0, &v_full[s]);
      } else if (sgk) {
        gather(vd, sgk->v + seg_off, VLO ? sgk->v_lo + seg_off : nullptr, nullptr, b * kKeys, pf_keys, &v_full[s]);
      } else {
        if (lane == 0) tma_block(vd, &tmV, VLO ? &tmVlo : nullptr, b, &v_full[s]);
      }
      ++vissued[s];
      __syncwarp();
    }
  } else if (warp == 1 || warp == 6) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues S = Q K^T, warp 6 O += P V, each in block order as soon as
    // its inputs are ready (the barriers order the two as a single issuer
    // would).  A tcgen05.mma holds its issuing thread for tens of cycles, so
    // one thread issuing both kept the next block's S waiting behind this
    // block's P V.
    const bool is_s = warp == 1;
    if (is_s) named_barrier_sync(1, 160);  // the rows past the Q box are zeroed
    if (lane == 0) {
      bool ok = true;
      if (is_s) {
        ok = mbar_wait(q_full, 0, wait_ns);
        if (!ok) fail(DEV_WAIT_TIMEOUT_MMA);
      }
      tc_fence_after_sync();
      constexpr uint32_t kIdescS = idesc_f16_f32(kRows, kKeys);
      constexpr uint32_t kIdescO = idesc_f16_f32(kRows, kDH) | (1u << 16);  // B (V) is MN-major
      const uint32_t qa = smem_u32(smem + kOffQ);
      int n = 0;
      uint64_t t_last = globaltimer_ns();
      uint32_t spins = 0;
      while (ok && n < my_n) {
        const int s = n % kStages;
        const uint32_t par = static_cast<uint32_t>((n / kStages) & 1);
        bool ready;
        if (is_s) {
          // S/P columns s are free once the P V of block n - kStages is done
          ready = mbar_test(&k_full[s], par) &&
                  (n < kStages || mbar_test(&pv_done[s], static_cast<uint32_t>(((n - kStages) / kStages) & 1)));
          if (ready) {
            tc_fence_after_sync();
            const uint32_t ka = smem_u32(smem + kOffK + s * kKSt);
            const uint32_t dS = tbase + kColS + s * kKeys;
#pragma unroll
            for (int k = 0; k < kDH / 16; ++k) {
              const uint32_t qo = (k >> 2) * (kQBytes / 2) + (k & 3) * 32, ko = (k >> 2) * (kKVBytes / 2) + (k & 3) * 32;
              umma_f16(dS, sdesc_kmajor_sw128(qa + qo), sdesc_kmajor_sw128(ka + ko), kIdescS, k > 0 ? 1u : 0u);
              if constexpr (QLO) {  // + Q K_lo + Q_lo K (the lo x lo term is below fp32 resolution of S)
                umma_f16(dS, sdesc_kmajor_sw128(qa + qo), sdesc_kmajor_sw128(ka + kKVBytes + ko), kIdescS, 1u);
                umma_f16(dS, sdesc_kmajor_sw128(qa + kQBytes + qo), sdesc_kmajor_sw128(ka + ko), kIdescS, 1u);
              }
            }
            umma_commit(&s_full[s]);
            umma_commit(&k_free[s]);
          }
        } else {
          ready = mbar_test(&p_full[s], par) && mbar_test(&v_full[s], par);
          if (ready) {
            tc_fence_after_sync();
            const uint32_t va = smem_u32(smem + kOffV + s * kVSt);
            const uint32_t pcol = tbase + kColS + s * kKeys;
#pragma unroll
            for (int k = 0; k < kKeys / 16; ++k) {  // P: 16 keys = 8 packed columns per step
              umma_f16_ts(tbase + kColO, pcol + k * 8, sdesc_mnmajor_sw128(va + k * 16 * 128, kKVBytes / 2, 1024), kIdescO,
                          (n > 0 || k > 0) ? 1u : 0u);
              if constexpr (VLO) {  // + P V_lo + P_lo V
                umma_f16_ts(tbase + kColO, pcol + k * 8,
                            sdesc_mnmajor_sw128(va + kKVBytes + k * 16 * 128, kKVBytes / 2, 1024), kIdescO, 1u);
                umma_f16_ts(tbase + kColO, pcol + 32 + k * 8, sdesc_mnmajor_sw128(va + k * 16 * 128, kKVBytes / 2, 1024),
                            kIdescO, 1u);
              }
            }
            umma_commit(&pv_done[s]);
            umma_commit(&v_free[s]);
          }
        }
        if (ready) {
          ++n;
          t_last = globaltimer_ns();
          continue;
        }
        __nanosleep(32);  // leave the issue slots to the softmax warp that shares this scheduler
        if ((++spins & 63) == 0) {
          if (*abort_flag) break;
          if (globaltimer_ns() - t_last > wait_ns) {
            fail(DEV_WAIT_TIMEOUT_MMA);
            break;
          }
        }
      }
      // every MMA this thread issued has finished before TMEM is released
      uint64_t* dr = is_s ? drain : drain2;
      umma_commit(dr);
      if (!mbar_wait(dr, 0, kDrainWaitNs)) record_error(err, DEV_WAIT_TIMEOUT_DRAIN);
    }
    __syncwarp();
  } else if (warp <= 5) {
    // ------------------------------------------------------------ softmax rows
    {  // the Q tile arrives by TMA (rows tt * G + g); the rows past it are zero
      if (r >= a.tpt * G) {
#pragma unroll 1
        for (int part = 0; part < (QLO ? 2 : 1); ++part)
#pragma unroll
          for (int c = 0; c < 16; ++c)
            *reinterpret_cast<uint4*>(smem + kOffQ + part * kQBytes + (c >> 3) * (kQBytes / 2) + swz(r, c & 7)) =
                make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
    }
    named_barrier_sync(1, 160);
    const uint32_t trow = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const bool valid = r < rows;
    // padding rows (r >= rows) take the same path as the tile's last token: their Q is zero and
    // their output is never written, and keeping the warp on one path keeps it in step
    const int pos = branch ? INT_MAX : a.pf_pos0 + t0 + r / G;
    const int tt = valid ? r / G : 0;
    // the visibility mask of the tile's first ancestor chunk, loaded ahead
    const unsigned long long mk0 = (valid && nb > nbp) ? a.tile_mask[static_cast<size_t>(ch0) * a.tpt + tt] : 0ull;
    for (int i = 0; i < my_n; ++i) {
      const int s = i % kStages, b = block_of(i);
      const bool ok = __all_sync(0xffffffffu, !*abort_flag &&
                                                  mbar_wait(&s_full[s], static_cast<uint32_t>((i / kStages) & 1), wait_ns));
      if (!ok) {
        if (lane == 0) fail(DEV_WAIT_TIMEOUT_MMA);
        break;
      }
      tc_fence_after_sync();
      float sv[kKeys];
      tmem_ld_32cols(trow + kColS + s * kKeys, sv);
      tmem_ld_32cols(trow + kColS + s * kKeys + 32, sv + 32);

      const bool local = b >= nbp;
      const int j0 = b * kKeys;
      // a prefix block wholly below the causal edge needs no per-key test
      const bool all_vis = !local && j0 + kKeys <= pf_keys && j0 + kKeys - 1 <= pos;
      float mb = -INFINITY;
      if (all_vis) {
#pragma unroll
        for (int c = 0; c < kKeys; ++c) mb = fmaxf(mb, sv[c]);
      } else {
        unsigned long long mk = 0ull;
        if (local && valid) mk = b == nbp ? mk0 : a.tile_mask[static_cast<size_t>(ch0 + b - nbp) * a.tpt + tt];
#pragma unroll
        for (int c = 0; c < kKeys; ++c) {
          const bool vis = local ? ((mk >> c) & 1ull) != 0ull : (j0 + c < pf_keys && j0 + c <= pos);
          sv[c] = vis ? sv[c] : -INFINITY;
          mb = fmaxf(mb, sv[c]);
        }
      }
      mb *= a.scale_log2;  // log2 units; -inf stays -inf
      if (__any_sync(0xffffffffu, mb > m_ref + kRescale)) {
        const float m_new = fmaxf(m_ref, mb);
        const float f = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - m_new);
        if (i > 0) {  // O holds blocks 0 .. i-1 once their last P V is done
          if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[(i - 1) % kStages],
                                                 static_cast<uint32_t>(((i - 1) / kStages) & 1), wait_ns))) {
            if (lane == 0) fail(DEV_WAIT_TIMEOUT_MMA);
            break;
          }
          tc_fence_after_sync();
#pragma unroll 1
          for (int q = 0; q < kDH / 32; ++q) {
            float ov[32];
            tmem_ld_32cols(trow + kColO + q * 32, ov);
#pragma unroll
            for (int x = 0; x < 32; ++x) ov[x] *= f;
            tmem_st_32cols(trow + kColO + q * 32, ov);
          }
        }
        l *= f;
        m_ref = m_new;
      }
      // P (fp16, two keys per column) over the first half of this block's S columns
      const float mo = (m_ref == -INFINITY) ? 0.f : m_ref;  // nothing visible yet: every score is -inf
      float ps = 0.f;
      uint32_t pw[kKeys / 2];
#pragma unroll
      for (int c2 = 0; c2 < kKeys / 2; ++c2) {
        const float p0 = ex2_approx(fmaf(sv[2 * c2], a.scale_log2, -mo));  // 2^-inf = 0
        const float p1 = ex2_approx(fmaf(sv[2 * c2 + 1], a.scale_log2, -mo));
        ps += p0 + p1;
        pw[c2] = pack2(p0, p1);
        if constexpr (VLO) {  // the remainders, kept in sv for the second store
          const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&pw[c2]));
          sv[2 * c2] = p0 - h.x;
          sv[2 * c2 + 1] = p1 - h.y;
        }
      }
      tmem_st_32cols_u32(trow + kColS + s * kKeys, pw);
      if constexpr (VLO) {
#pragma unroll
        for (int c2 = 0; c2 < kKeys / 2; ++c2) pw[c2] = pack2(sv[2 * c2], sv[2 * c2 + 1]);
        tmem_st_32cols_u32(trow + kColS + s * kKeys + 32, pw);
      }
      l += ps;
      tc_fence_before_sync();
      mbar_arrive(&p_full[s]);
    }
    have_o = my_n > 0 && !*abort_flag;
    if (have_o && !mbar_wait(&pv_done[(my_n - 1) % kStages], static_cast<uint32_t>(((my_n - 1) / kStages) & 1),
                             wait_ns)) {
      if (lane == 0) fail(DEV_WAIT_TIMEOUT_MMA);
      have_o = false;
    }
    have_o = __all_sync(0xffffffffu, have_o);
    tc_fence_after_sync();
    if (csk == 1) {
      // normalised rows staged in shared memory (every MMA is done: Q, K and V
      // are free), then one bulk copy per 256-byte output row
      const float il = l > 0.f ? 1.f / l : 0.f;
      uint8_t* shi = smem + r * kOutLd;
      uint8_t* slo = smem + (kRows + r) * kOutLd;
#pragma unroll 1
      for (int q = 0; q < kDH / 32 && have_o; ++q) {
        float ov[32];
        tmem_ld_32cols(trow + kColO + q * 32, ov);
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t w[4], wl[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const float y0 = ov[c8 * 8 + 2 * x] * il, y1 = ov[c8 * 8 + 2 * x + 1] * il;
            w[x] = pack2(y0, y1);
            const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&w[x]));
            wl[x] = pack2(y0 - h.x, y1 - h.y);
          }
          *reinterpret_cast<uint4*>(shi + q * 64 + c8 * 16) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(slo + q * 64 + c8 * 16) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        }
      }
      // the four softmax warps copy the staged rows out together: a token's G
      // rows are adjacent in the output, so 16 lanes write one 256-byte row
      // and a warp two rows per store
      named_barrier_sync(2, 128);
      if (my_n > 0 && !*abort_flag) {
        const int tid = threadIdx.x - 64;  // softmax threads: warps 2-5
        const int per_part = rows * 16;
        const int n_idx = (a.out_lo ? 2 : 1) * per_part;
        for (int idx = tid; idx < n_idx; idx += 128) {
          const int part = idx >= per_part ? 1 : 0;
          const int rem = idx - part * per_part;
          const int rr = rem >> 4, c = rem & 15;
          const uint4 v = *reinterpret_cast<const uint4*>(smem + (part * kRows + rr) * kOutLd + c * 16);
          act_t* dst = (part ? a.out_lo : a.out) + static_cast<size_t>(qrow0 + rr / G) * a.ld_out +
                       (hk * G + rr % G) * kDH;
          *reinterpret_cast<uint4*>(dst + c * 8) = v;
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    // nothing of this CTA's copies may still be landing when it exits
    mbar_wait(q_full, 0, kDrainWaitNs);
    for (int s = 0; s < kStages; ++s) {
      if (kissued[s] > 0) mbar_wait(&k_full[s], static_cast<uint32_t>((kissued[s] - 1) & 1), kDrainWaitNs);
      if (vissued[s] > 0) mbar_wait(&v_full[s], static_cast<uint32_t>((vissued[s] - 1) & 1), kDrainWaitNs);
    }
  }
  if (csk > 1) {
    // rank q owns rows [q * per, (q + 1) * per) of the tile: every CTA pushes
    // its partial state of those rows (unnormalised O relative to its m, and
    // its l) into slot `rank` of the owner's shared memory, then the owner
    // combines them locally
    const int per = (kRows + csk - 1) / csk;
    cluster_sync_all();  // every CTA of the cluster is done with its Q/K/V/P buffers
    if (warp >= 2 && warp <= 5) {
      const uint32_t trow = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
      const int owner = r / per, lr = r - owner * per;
      const uint32_t dst = dsmem_addr(sRed + (rank * per + lr) * kRedLd, owner);
#pragma unroll 1
      for (int q = 0; q < kDH / 32; ++q) {
        float ov[32];
        if (have_o) {
          tc_fence_after_sync();
          tmem_ld_32cols(trow + kColO + q * 32, ov);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) ov[x] = 0.f;
        }
        if (r < rows)
#pragma unroll
          for (int x = 0; x < 8; ++x)
            dsmem_st_f4(dst + (q * 32 + 4 * x) * 4, make_float4(ov[4 * x], ov[4 * x + 1], ov[4 * x + 2], ov[4 * x + 3]));
      }
      if (r < rows)
        dsmem_st_f2(dsmem_addr(sML + rank * per + lr, owner),
                    make_float2(have_o ? m_ref : -INFINITY, have_o ? l : 0.f));
    }
    tc_fence_before_sync();
    cluster_sync_all();  // the pushed states are visible to their owners
    const int rb = rank * per, re = min(rows, rb + per);
    constexpr int C4 = kDH / 4;
    for (int idx = threadIdx.x; idx < (re - rb) * C4; idx += blockDim.x) {
      const int lr = idx / C4, rr = rb + lr, d = (idx % C4) * 4;
      float M = -INFINITY;
      for (int pr = 0; pr < csk; ++pr) {
        const float2 ml = sML[pr * per + lr];
        if (ml.y > 0.f) M = fmaxf(M, ml.x);
      }
      float L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int pr = 0; pr < csk; ++pr) {
        const float2 ml = sML[pr * per + lr];
        if (!(ml.y > 0.f)) continue;
        const float w = ex2_approx(ml.x - M);
        const float4 v = *reinterpret_cast<const float4*>(sRed + (pr * per + lr) * kRedLd + d);
        L += w * ml.y;
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
      }
      const float il = L > 0.f ? 1.f / L : 0.f;
      const float y0 = acc.x * il, y1 = acc.y * il, y2 = acc.z * il, y3 = acc.w * il;
      const size_t o = static_cast<size_t>(qrow0 + rr / G) * a.ld_out + (hk * G + rr % G) * kDH + d;
      const uint2 hv = make_uint2(pack2(y0, y1), pack2(y2, y3));
      *reinterpret_cast<uint2*>(a.out + o) = hv;
      if (a.out_lo) {
        const float2 h01 = __half22float2(*reinterpret_cast<const __half2*>(&hv.x));
        const float2 h23 = __half22float2(*reinterpret_cast<const __half2*>(&hv.y));
        *reinterpret_cast<uint2*>(a.out_lo + o) = make_uint2(pack2(y0 - h01.x, y1 - h01.y), pack2(y2 - h23.x, y3 - h23.y));
      }
    }
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

template <bool QLO, bool VLO>
static int launch_tc_t(const TreeAttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmKlo,
                       const CUtensorMap& tmVlo, const CUtensorMap& tmQ, const CUtensorMap& tmQlo, int layer,
                       uint64_t wait_ns, int* err, cudaStream_t s) {
  using C = TcCfg<QLO, VLO>;
  static bool attr = false;
  if (!attr) {
    cudaError_t r =
        cudaFuncSetAttribute(tree_attn_tc_kernel<QLO, VLO>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (r != cudaSuccess) return r;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((a.n_br_tiles + a.n_pf_tiles) * a.csk), static_cast<unsigned>(a.Hkv), 1);
  cfg.blockDim = dim3(224, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int na = 0;
  if (a.csk > 1) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = static_cast<unsigned>(a.csk);
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl_enabled()) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, tree_attn_tc_kernel<QLO, VLO>, tmK, tmV, tmKlo, tmVlo, tmQ, tmQlo, a, layer, wait_ns, err);
}

int tree_attention_tc_slots(int csk) {
  // clusters must fit inside one GPC, so fewer CTAs than SMs may be resident
  // at once for csk > 1 (e.g. clusters of 5 on GPCs of 19 SMs)
  static int cache[9] = {};
  if (csk < 1 || csk > 8) return 0;
  if (cache[csk]) return cache[csk];
  // every variant runs one CTA per SM; the largest one's footprint decides
  using C = TcCfg<true, true>;
  auto kern = tree_attn_tc_kernel<true, true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess) return 0;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int slots = 0;
  if (csk == 1) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 224, C::kSmem) != cudaSuccess) return 0;
    slots = per_sm * sms;
  } else {
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(static_cast<unsigned>(csk * std::max(1, sms / csk)), 1, 1);
    q.blockDim = dim3(224, 1, 1);
    q.dynamicSmemBytes = C::kSmem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = static_cast<unsigned>(csk);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    q.attrs = at;
    q.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    slots = n * csk;
  }
  cache[csk] = slots;
  return slots;
}

int launch_tree_attention_tc(const TreeAttnArgs& a, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const CUtensorMap* tmKlo, const CUtensorMap* tmVlo, int layer, uint64_t wait_ns, int* err,
                             cudaStream_t s) {
  if (a.n_br_tiles + a.n_pf_tiles <= 0) return 0;
  if (a.DH != kDH || a.csk < 1 || a.csk > 8) return cudaErrorInvalidValue;
  if (a.tpt < 1 || a.tpt * (a.Hq / a.Hkv) > kRows) return cudaErrorInvalidValue;
  const bool lo = a.q_lo != nullptr;
  if (lo && (!tmKlo || !tmVlo || (a.n_br_tiles > 0 && (!a.kb_lo || !a.vb_lo)))) return cudaErrorInvalidValue;
  const bool qlo = lo && (a.lo_terms & 1) != 0, vlo = lo && (a.lo_terms & 2) != 0;
  // the Q tiles by TMA: the q rows hold every head of a token side by side
  const int G = a.Hq / a.Hkv;
  const int q_rows = std::max(a.n_pf, a.n_br_tiles > 0 ? a.br_row0 + a.n_br : 0);
  CUtensorMap mq, mql;
  if (!make_q_map(&mq, a.q, kDH, a.Hq, std::max(q_rows, 1), G, a.tpt)) return cudaErrorInvalidValue;
  if (qlo) {
    if (!make_q_map(&mql, a.q_lo, kDH, a.Hq, std::max(q_rows, 1), G, a.tpt)) return cudaErrorInvalidValue;
    if (vlo) return launch_tc_t<true, true>(a, tmK, tmV, *tmKlo, *tmVlo, mq, mql, layer, wait_ns, err, s);
    return launch_tc_t<true, false>(a, tmK, tmV, *tmKlo, tmV, mq, mql, layer, wait_ns, err, s);
  }
  if (vlo) return launch_tc_t<false, true>(a, tmK, tmV, tmK, *tmVlo, mq, mq, layer, wait_ns, err, s);
  return launch_tc_t<false, false>(a, tmK, tmV, tmK, tmV, mq, mq, layer, wait_ns, err, s);
}

}  // namespace pcd
