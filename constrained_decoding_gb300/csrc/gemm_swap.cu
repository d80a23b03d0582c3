// Weight-streaming GEMM for short activations (the branch pass's few hundred
// token rows): D^T[Nw][T] = W[Nw][K] . X[T][K]^T on a pair of CTAs sharing
// one tcgen05 MMA of M = 256 (cta_group::2).
//
// With the tokens as the MMA's M side (the ordinary orientation) every
// 128-row token tile pulls every weight tile into its own SM's shared memory,
// so a 313-row pass fills three times the weights from L2.  Here the weights
// are the 256-row side, split 128 rows per CTA, and the tokens are the MMA's
// N side (up to 512, as one or two pieces of at most 256), each CTA holding
// half of every piece: a k block brings 16 KB of weights plus T/2 token rows
// (x 128 bytes, twice with the activation remainder) into each SM, and every
// weight byte is read from HBM once.  The accumulator is T columns of fp32
// per TMEM lane (lane = weight row), double-buffered when T <= 256.
//
// Warps (both CTAs): 0 TMA producer (own 128 weight rows, own half of the
// token rows; completion on the leader's barrier), 1 TMEM allocation and, in
// the leader, the MMA issuer, 2-5 epilogue (each its 32-lane quarter of its
// CTA's accumulator rows, one 32-token chunk at a time).  Epilogues:
//   EPI_F32_ADD / EPI_F32_ATOMIC  out[t][n] += D^T[n][t]  (fp32; atomics for split K)
//   EPI_SWIGLU  rows (2f, 2f+1) = (gate_f, up_f): out[t][f] = silu(gate) * up, fp16
//               (adjacent lanes swap one value per token pair through a shuffle)
// Every wait is bounded.  On the way out the leader completes the stage
// barriers for every copy either CTA issued (both report what they issued),
// so no copy can land in a CTA that has exited.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>

#include "common.cuh"
#include "gemm.h"
#include "ptx.cuh"

namespace pcd {

struct SwapParams {
  int Nw, T, K;      // weight rows, token rows, depth
  int TP;            // tokens padded to 32: the MMA's N, in `np` pieces of TP / np
  int np;
  int n_pt, k_splits, n_units, nkb;
  int stages;
  uint32_t a_bytes;  // one CTA's weight tile per stage (128 rows x 128 B)
  uint32_t b_bytes;  // one CTA's token rows per stage and operand part (TP / 2 x 128 B)
  uint32_t part;     // bytes one CTA loads per stage
  uint64_t wait_ns;
  int* err;
  int a_const;       // weight tiles may load before the programmatic dependency wait
};

constexpr int kSwapBarOff = 0;  // barriers at the start of the aligned shared memory
constexpr int kSwapHdr = 1024;  // barrier block; the stages follow, 1024-aligned

template <int EPI, bool BLO>
__global__ void __launch_bounds__(192, 1)
    gemm_swap_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmXlo, const SwapParams p, const EpiArgs e) {
  extern __shared__ uint8_t swap_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(swap_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSwapBarOff);  // [8], leader's are used
  uint64_t* empty = full + 8;                                         // [8], both CTAs
  uint64_t* tfull = empty + 8;                                        // [2], both CTAs
  uint64_t* tempty = tfull + 2;                                       // [2], leader's are used
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* peer_cnt = reinterpret_cast<uint32_t*>(smem + 512);    // [8] the peer's issued phases per stage
  uint32_t* peer_last = peer_cnt + 8;                              // [8] bytes of its last phase
  uint8_t* stages = smem + kSwapHdr;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int pair = static_cast<int>(cluster_id_x());
  const int n_pairs = static_cast<int>(n_clusters_x());
  const int S = p.stages;
  const int acc_stages = (2 * p.TP <= 512) ? 2 : 1;
  const int NPc = p.TP / p.np;  // columns of one MMA piece

  if (threadIdx.x == 0) {
    for (int s = 0; s < 8; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 256);  // every epilogue thread of both CTAs
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    if constexpr (BLO) tma_prefetch_desc(&tmXlo);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync_all();  // both CTAs' barriers exist before either signals the other
  tc_fence_after_sync();
  const uint32_t tbase = *tmem_slot;

  auto unit = [&](int u, int& pt, int& kb0, int& kb1) {
    pt = u / p.k_splits;
    const int ks = u - pt * p.k_splits;
    kb0 = ks * p.nkb / p.k_splits;
    kb1 = (ks + 1) * p.nkb / p.k_splits;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    uint32_t cnt[8], last[8];  // phases this CTA issued into each stage, bytes of the last one
    for (int s = 0; s < 8; ++s) cnt[s] = 0, last[s] = 0;
    if (lane == 0) {
      const uint32_t fb0 = cluster_addr(&full[0], 0);
      auto fbar = [&](int s) { return fb0 + static_cast<uint32_t>(s) * 8u; };
      auto load_w = [&](int s, int pt, int kb) {
        if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * p.part);
        tma_load_2d_pair(stages + static_cast<size_t>(s) * p.part, &tmW, fbar(s), kb * 64, pt * 256 + rank * 128);
        cnt[s] += 1;
        last[s] = p.a_bytes;
      };
      auto load_x = [&](int s, int kb) {
        uint8_t* b = stages + static_cast<size_t>(s) * p.part + p.a_bytes;
        for (int j = 0; j < p.np; ++j) {
          const int row = j * NPc + rank * (NPc / 2);
          tma_load_2d_pair(b + j * (NPc / 2) * 128, &tmX, fbar(s), kb * 64, row);
          if constexpr (BLO) tma_load_2d_pair(b + p.b_bytes + j * (NPc / 2) * 128, &tmXlo, fbar(s), kb * 64, row);
        }
        last[s] += (BLO ? 2u : 1u) * p.b_bytes;
      };
      // the weights do not depend on earlier kernels: the first ring of
      // stages gets its weight tiles before the dependency wait
      int pre = 0;
      if (p.a_const) {
        for (int u = pair; u < p.n_units && pre < S; u += n_pairs) {
          int pt, kb0, kb1;
          unit(u, pt, kb0, kb1);
          for (int kb = kb0; kb < kb1 && pre < S; ++kb, ++pre) load_w(pre, pt, kb);
        }
      }
      griddep_launch_dependents();
      griddep_wait();
      int stage = 0, it = 0;
      uint32_t phase = 0;
      for (int u = pair; u < p.n_units && !*abort_flag; u += n_pairs) {
        int pt, kb0, kb1;
        unit(u, pt, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          if (it >= pre) {
            if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns)) {
              record_error(p.err, DEV_WAIT_TIMEOUT_PRODUCER);
              *abort_flag = 1;
              break;
            }
            load_w(stage, pt, kb);
          }
          load_x(stage, kb);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (rank == 1) {
        // report what this CTA issued to the leader, which completes the drain
        for (int s = 0; s < S; ++s) {
          asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr(&peer_cnt[s], 0)), "r"(cnt[s])
                       : "memory");
          asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr(&peer_last[s], 0)), "r"(last[s])
                       : "memory");
        }
      }
    } else {
      griddep_launch_dependents();
      griddep_wait();
    }
    tc_fence_before_sync();
    cluster_sync_all();  // (1) no copy is issued after this
    if (lane == 0 && rank == 0) {
      // every phase either CTA issued into, completed: expected bytes that
      // were never issued are counted as done, a phase the peer issued ahead
      // of this CTA's arming is armed with the peer's bytes
      for (int s = 0; s < S; ++s) {
        const uint32_t a = cnt[s], n = peer_cnt[s], pb = peer_last[s];
        if (a == 0 && n == 0) continue;
        if (n > a + 1 || n + 1 < a) {  // cannot happen: each CTA's ring waits on the other's previous phase
          record_error(p.err, DEV_WAIT_TIMEOUT_DRAIN);
          continue;
        }
        uint32_t ph_last;
        if (n == a + 1) {
          mbar_arrive_expect_tx(&full[s], pb);
          ph_last = n - 1;
        } else {
          const uint32_t owed = (p.part - last[s]) + (n == a ? p.part - pb : p.part);
          if (owed) mbar_complete_tx(&full[s], owed);
          ph_last = a - 1;
        }
        if (!mbar_wait(&full[s], ph_last & 1u, kDrainWaitNs)) record_error(p.err, DEV_WAIT_TIMEOUT_DRAIN);
      }
    }
  } else if (warp == 1) {
    griddep_launch_dependents();
    griddep_wait();
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = idesc_f16_f32(256, NPc);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool any = false;
      for (int u = pair; u < p.n_units && !*abort_flag; u += n_pairs) {
        int pt, kb0, kb1;
        unit(u, pt, kb0, kb1);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, p.wait_ns)) {
          record_error(p.err, DEV_WAIT_TIMEOUT_MMA);
          *abort_flag = 1;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_base = tbase + static_cast<uint32_t>(acc * p.TP);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.wait_ns)) {
            record_error(p.err, DEV_WAIT_TIMEOUT_MMA);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_base = smem_u32(stages + static_cast<size_t>(stage) * p.part);
          const uint32_t b_base = a_base + p.a_bytes;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = sdesc_kmajor_sw128(a_base + k * 32);
            for (int j = 0; j < p.np; ++j) {
              const uint32_t bj = b_base + static_cast<uint32_t>(j * (NPc / 2) * 128 + k * 32);
              umma_f16_pair(d_base + j * NPc, ad, sdesc_kmajor_sw128(bj), idesc, (kb > kb0 || k > 0) ? 1u : 0u);
              if constexpr (BLO) umma_f16_pair(d_base + j * NPc, ad, sdesc_kmajor_sw128(bj + p.b_bytes), idesc, 1u);
            }
          }
          umma_commit_pair_mc(&empty[stage]);  // both CTAs' stage is free once these MMAs are done
          any = true;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(&tfull[acc]);
        if (++acc == acc_stages) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (any) {
        umma_commit_pair(drain);
        if (!mbar_wait(drain, 0, kDrainWaitNs)) record_error(p.err, DEV_WAIT_TIMEOUT_DRAIN);
      }
    }
    tc_fence_before_sync();
    cluster_sync_all();  // (1)
  } else {
    griddep_launch_dependents();
    griddep_wait();
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = pair; u < p.n_units && !*abort_flag; u += n_pairs) {
      int pt, kb0, kb1;
      unit(u, pt, kb0, kb1);
      if (!mbar_wait(&tfull[acc], acc_phase, p.wait_ns)) {
        record_error(p.err, DEV_WAIT_TIMEOUT_EPILOGUE);
        *abort_flag = 1;
        break;
      }
      tc_fence_after_sync();
      const int n = pt * 256 + rank * 128 + q * 32 + lane;  // weight row of this thread's TMEM lane
      const bool nv = n < p.Nw;
      const uint32_t t_row = tbase + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * p.TP);
      for (int c0 = 0; c0 < p.T; c0 += 32) {
        float v[32];
        tmem_ld_32cols(t_row + c0, v);
        if constexpr (EPI == EPI_F32_ADD || EPI == EPI_F32_ATOMIC) {
          if (nv) {
            float* o = reinterpret_cast<float*>(e.out) + static_cast<size_t>(c0) * e.ldo + n;
            const int nt = min(32, p.T - c0);
            if constexpr (EPI == EPI_F32_ATOMIC) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < nt) atomicAdd(o + static_cast<size_t>(i) * e.ldo, v[i]);
            } else {
              // all loads first: the stores could alias later loads, which
              // would otherwise serialise every read-modify-write
              float r[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = i < nt ? o[static_cast<size_t>(i) * e.ldo] : 0.f;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < nt) o[static_cast<size_t>(i) * e.ldo] = r[i] + v[i];
            }
          }
        } else if constexpr (EPI == EPI_SWIGLU) {
          const bool odd = lane & 1;
          const int f = n >> 1;
          act_t* o = reinterpret_cast<act_t*>(e.out);
          act_t* ol = reinterpret_cast<act_t*>(e.out_lo);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            // even lane: gate_f at tokens 2j, 2j+1; odd lane: up_f.  The even
            // lane finishes token 2j, the odd one token 2j + 1.
            const float send = odd ? v[2 * j] : v[2 * j + 1];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const float h = odd ? silu_f(recv) * v[2 * j + 1] : silu_f(v[2 * j]) * recv;
            const int t = c0 + 2 * j + (odd ? 1 : 0);
            if (nv && t < p.T) {
              const size_t off = static_cast<size_t>(t) * e.ldo + f;
              const act_t hv = f2a(h);
              o[off] = hv;
              if (ol) ol[off] = f2a(h - a2f(hv));
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive_cluster(cluster_addr(&tempty[acc], 0));  // the leader may reuse the accumulator
      if (++acc == acc_stages) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    tc_fence_before_sync();
    cluster_sync_all();  // (1)
  }

  tc_fence_before_sync();
  cluster_sync_all();  // (2) the leader has seen every copy land; TMEM is idle
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tbase, 512);
  }
}

// ====================================================================== host
int swap_stage_count(int TP, bool blo) {
  const int part = 16384 + (blo ? 2 : 1) * (TP / 2) * 128;
  const int budget = 227 * 1024 - kSwapHdr - 1024;
  return std::min(8, budget / part);
}

template <int EPI, bool BLO>
static int launch_swap_t(const CUtensorMap& mw, const CUtensorMap& mx, const CUtensorMap& mxl, const SwapParams& p,
                         const EpiArgs& e, cudaStream_t st, int sms) {
  auto kern = gemm_swap_kernel<EPI, BLO>;
  const size_t smem = static_cast<size_t>(kSwapHdr) + static_cast<size_t>(p.stages) * p.part + 1024;
  static int max_pairs = 0;  // per instantiation: the kernel is persistent, one pair per two SMs
  if (!max_pairs) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (r != cudaSuccess) return r;
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(2 * (sms / 2), 1, 1);
    q.blockDim = dim3(192, 1, 1);
    q.dynamicSmemBytes = 227 * 1024;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    q.attrs = at;
    q.numAttrs = 1;
    int n = 0;
    r = cudaOccupancyMaxActiveClusters(&n, kern, &q);
    if (r != cudaSuccess) return r;
    max_pairs = n > 0 ? n : 1;
  }
  const int pairs = std::min(p.n_units, max_pairs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  int na = 1;
  if (pdl_enabled()) {
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    na = 2;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, mw, mx, mxl, p, e);
}

int swap_max_pairs(int sms) { return std::max(1, sms / 2); }

int swap_splits(int Nw, int K, int epi, int sms) {
  const int n_pt = ceil_div(Nw, 256), nkb = K / 64;
  if (epi != EPI_F32_ATOMIC) return 1;
  const int pairs = swap_max_pairs(sms);
  // fill the pairs, keeping at least four k blocks per unit
  int sp = std::max(1, pairs / n_pt);
  sp = std::min(sp, std::max(1, nkb / 4));
  return sp;
}

int launch_gemm_swap(const SwapShape& s, int epi, const EpiArgs& e, int splits, cudaStream_t stream, int* dev_err,
                     uint64_t wait_ns, int sms) {
  const int Nw = s.w_rows, T = s.x_rows, K = s.K;
  if (T <= 0 || Nw <= 0) return 0;
  if (T > kSwapMaxRows || K <= 0 || K % 64 || Nw % 32) return -1;
  if (epi != EPI_F32_ADD && epi != EPI_F32_ATOMIC && epi != EPI_SWIGLU) return -1;
  if (splits > 1 && epi != EPI_F32_ATOMIC) return -1;
  SwapParams p;
  p.Nw = Nw;
  p.T = T;
  p.K = K;
  p.TP = ceil_div(T, 32) * 32;
  p.np = p.TP > 256 ? 2 : 1;
  p.nkb = K / 64;
  p.n_pt = ceil_div(Nw, 256);
  p.k_splits = std::max(1, std::min(splits, p.nkb));
  p.n_units = p.n_pt * p.k_splits;
  p.a_bytes = 128 * 128;
  p.b_bytes = static_cast<uint32_t>(p.TP / 2) * 128;
  const bool blo = s.x_lo != nullptr;
  p.part = p.a_bytes + (blo ? 2u : 1u) * p.b_bytes;
  p.stages = swap_stage_count(p.TP, blo);
  if (p.stages < 2) return -1;
  p.wait_ns = wait_ns;
  p.err = dev_err;
  p.a_const = s.w_const ? 1 : 0;
  CUtensorMap mw, mx, mxl;
  const int box_x = (p.TP / p.np) / 2;
  if (!make_tile_map(&mw, s.w, Nw, K, s.w_ld, 128)) return -1;
  if (!make_tile_map(&mx, s.x, T, K, s.x_ld, box_x)) return -1;
  if (blo) {
    if (!make_tile_map(&mxl, s.x_lo, T, K, s.x_ld, box_x)) return -1;
  } else {
    mxl = mx;
  }
  switch (epi) {
    case EPI_F32_ADD:
      return blo ? launch_swap_t<EPI_F32_ADD, true>(mw, mx, mxl, p, e, stream, sms)
                 : launch_swap_t<EPI_F32_ADD, false>(mw, mx, mxl, p, e, stream, sms);
    case EPI_F32_ATOMIC:
      return blo ? launch_swap_t<EPI_F32_ATOMIC, true>(mw, mx, mxl, p, e, stream, sms)
                 : launch_swap_t<EPI_F32_ATOMIC, false>(mw, mx, mxl, p, e, stream, sms);
    case EPI_SWIGLU:
      return blo ? launch_swap_t<EPI_SWIGLU, true>(mw, mx, mxl, p, e, stream, sms)
                 : launch_swap_t<EPI_SWIGLU, false>(mw, mx, mxl, p, e, stream, sms);
  }
  return -1;
}

}  // namespace pcd
