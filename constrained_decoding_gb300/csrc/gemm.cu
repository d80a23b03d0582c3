// tcgen05 GEMM for sm_103a: D[M][N] = A[M][K] . B[N][K]^T, fp16 in, fp32
// accumulation in tensor memory (TMEM).
//
// One persistent CTA per SM, 6 warps:
//   warp 0     TMA producer: fills a ring of shared-memory stages, each holding
//              MT A tiles (128 x 64) and one B tile (BN x 64), 128-byte swizzled;
//   warp 1     allocates TMEM; one thread issues tcgen05.mma (M=128, N=BN,
//              K=16) for every A tile against the shared B tile, so one B tile
//              (the weights) read from HBM feeds MT*128 rows of A;
//   warps 2-5  epilogue: read the accumulator from TMEM (each warp owns one
//              32-lane quarter) and apply the fused epilogue.
// Accumulators are double-buffered in TMEM when MT*BN <= 256, so the epilogue
// of one work unit overlaps the main loop of the next.
// A work unit is (N tile, K split, group of MT M tiles), ordered so that the
// units sharing a B tile run on neighbouring CTAs at the same time and read
// it from L2.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>
#include <unordered_map>

#include "common.cuh"
#include "gemm.h"
#include "ptx.cuh"

namespace pcd {

struct GemmParams {
  int M, N, K;
  int n_mgroups, n_ntiles, k_splits, n_units, nkb;
  uint64_t wait_ns;
  int* err;
  int b_evict_first;  // B is read by one M group only: stream it past L2
  int lo_row0;        // ALO: tiles entirely below this row have no low half
  int b_const;        // B tiles may load before the programmatic dependency wait
  int n_wide;         // units of the full N tile width; units past it are 64-column slices of
  int nw_col0;        //   the last N tiles, from column nw_col0 (the last wave's tail, split finer)
};

template <int MT, int BN, bool ALO = false>
struct GemmCfg {
  static constexpr int A_BYTES = 128 * 128;  // 128 rows x 64 fp16
  static constexpr int B_BYTES = BN * 128;
  static constexpr int A_PARTS = ALO ? 2 : 1;  // A as hi + lo fp16 halves
  static constexpr int STAGE_BYTES = A_PARTS * MT * A_BYTES + B_BYTES;
  static constexpr int SMEM_BUDGET = 227 * 1024 - 2048;
  static constexpr int STAGES_RAW = SMEM_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int ACC_COLS = MT * BN;
  static constexpr int ACC_STAGES = (2 * ACC_COLS <= 512) ? 2 : 1;
  static constexpr int TMEM_COLS_RAW = ACC_STAGES * ACC_COLS;
  static constexpr int TMEM_COLS = TMEM_COLS_RAW <= 32    ? 32
                                   : TMEM_COLS_RAW <= 64  ? 64
                                   : TMEM_COLS_RAW <= 128 ? 128
                                   : TMEM_COLS_RAW <= 256 ? 256
                                                          : 512;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align slack*/ + 256 /*barriers*/;
  static_assert(ACC_STAGES * ACC_COLS <= 512, "accumulator does not fit in TMEM");
  static_assert(STAGES >= 2, "need at least two pipeline stages");
};

__device__ __forceinline__ void decode_unit(const GemmParams& p, int u, int& nt, int& mg, int& ks) {
  mg = u % p.n_mgroups;
  const int rest = u / p.n_mgroups;
  ks = rest % p.k_splits;
  nt = rest / p.k_splits;
}

template <int EPI>
__device__ __forceinline__ void epi_chunk(const GemmParams& p, const EpiArgs& e, int row, int col0, const float* v,
                                          float& run_m, float& run_s) {
  if constexpr (EPI == EPI_READOUT) {
    // online max / sum-exp over the valid vocabulary columns of this chunk
    float cm = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i < p.N) cm = fmaxf(cm, v[i]);
    const float nm = fmaxf(run_m, cm);
    float acc = (run_m == -INFINITY) ? 0.f : run_s * __expf(run_m - nm);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i < p.N) acc += __expf(v[i] - nm);
    run_m = nm;
    run_s = acc;
  } else {
    if (row >= p.M) return;
    if constexpr (EPI == EPI_BF16) {
      act_t* o = reinterpret_cast<act_t*>(e.out) + static_cast<size_t>(row) * e.ldo + col0;
      uint4* o4 = reinterpret_cast<uint4*>(o);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint4 w;
        w.x = pack2(v[8 * j + 0], v[8 * j + 1]);
        w.y = pack2(v[8 * j + 2], v[8 * j + 3]);
        w.z = pack2(v[8 * j + 4], v[8 * j + 5]);
        w.w = pack2(v[8 * j + 6], v[8 * j + 7]);
        o4[j] = w;
      }
    } else if constexpr (EPI == EPI_F32_ADD) {
      float4* o4 = reinterpret_cast<float4*>(reinterpret_cast<float*>(e.out) + static_cast<size_t>(row) * e.ldo + col0);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float4 a = o4[j];
        a.x += v[4 * j + 0];
        a.y += v[4 * j + 1];
        a.z += v[4 * j + 2];
        a.w += v[4 * j + 3];
        o4[j] = a;
      }
    } else if constexpr (EPI == EPI_F32_STORE) {
      float4* o4 = reinterpret_cast<float4*>(reinterpret_cast<float*>(e.out) + static_cast<size_t>(row) * e.ldo + col0);
#pragma unroll
      for (int j = 0; j < 8; ++j) o4[j] = make_float4(v[4 * j + 0], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    } else if constexpr (EPI == EPI_F32_ATOMIC) {
      float4* o4 = reinterpret_cast<float4*>(reinterpret_cast<float*>(e.out) + static_cast<size_t>(row) * e.ldo + col0);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        atomicAdd(o4 + j, make_float4(v[4 * j + 0], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
    } else if constexpr (EPI == EPI_SWIGLU) {
      act_t* o = reinterpret_cast<act_t*>(e.out) + static_cast<size_t>(row) * e.ldo + col0 / 2;
      uint4* o4 = reinterpret_cast<uint4*>(o);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = silu_f(v[16 * j + 2 * i]) * v[16 * j + 2 * i + 1];
        uint4 w;
        w.x = pack2(h[0], h[1]);
        w.y = pack2(h[2], h[3]);
        w.z = pack2(h[4], h[5]);
        w.w = pack2(h[6], h[7]);
        o4[j] = w;
        if (e.out_lo) {
          const __half* hh = reinterpret_cast<const __half*>(&w);
          uint4 lo;
          lo.x = pack2(h[0] - __half2float(hh[0]), h[1] - __half2float(hh[1]));
          lo.y = pack2(h[2] - __half2float(hh[2]), h[3] - __half2float(hh[3]));
          lo.z = pack2(h[4] - __half2float(hh[4]), h[5] - __half2float(hh[5]));
          lo.w = pack2(h[6] - __half2float(hh[6]), h[7] - __half2float(hh[7]));
          reinterpret_cast<uint4*>(reinterpret_cast<act_t*>(e.out_lo) + static_cast<size_t>(row) * e.ldo + col0 / 2)[j] = lo;
        }
      }
    }
  }
}

// Fused q/k/v epilogue: for each 128-wide head of the tile, the thread (one
// token row) rotates the pairs (i, i + 64) by the row's rotary angle
// (rotate-half pairing; cos/sin from a double-precision table) and writes q,
// or k and v, in fp16 straight to their destinations.
template <int BN>
__device__ __forceinline__ void epi_qkv_rope(const GemmParams& p, const EpiArgs& e, int row, int nt, uint32_t t_row) {
  const bool valid = row < p.M;
  const int dst = row >= e.split_row ? 1 : 0;
  const int r2 = row - (dst ? e.split_row : 0);
  int pos = 0;
  if (valid) {
    pos = e.pos_base[dst] + (e.pos_rel[dst] ? e.pos_rel[dst][r2] : r2);
    if (pos < 0 || pos >= e.max_pos) {
      record_error(e.err, DEV_BAD_INDEX);
      pos = 0;
    }
  }
  const float2* cs = e.rope_cs + pos;  // pair i at cs[i * max_pos]
#pragma unroll 1
  for (int hh = 0; hh < BN / 128; ++hh) {
    const int head = (nt * BN) / 128 + hh;
    if (head * 128 >= p.N) break;  // uniform across the warp
    const bool is_v = head >= e.n_q_heads + e.n_kv_heads;
    act_t* out;
    act_t* out_lo;  // the remainder's row, or nullptr
    if (head < e.n_q_heads) {
      const size_t o = static_cast<size_t>(row) * e.n_q_heads * 128 + head * 128;
      out = e.q_out + o;
      out_lo = e.q_lo ? e.q_lo + o : nullptr;
    } else {
      const int kh = is_v ? head - e.n_q_heads - e.n_kv_heads : head - e.n_q_heads;
      const size_t o = (static_cast<size_t>(kh) * e.kv_stride[dst] + e.kv_row0[dst] + r2) * 128;
      out = (is_v ? e.kv_v[dst] : e.kv_k[dst]) + o;
      act_t* lb = is_v ? e.kv_v_lo[dst] : e.kv_k_lo[dst];
      out_lo = lb ? lb + o : nullptr;
    }
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      float a[32], b[32];
      tmem_ld_32cols(t_row + hh * 128 + half * 32, a);
      tmem_ld_32cols(t_row + hh * 128 + 64 + half * 32, b);
      if (!valid) continue;
      if (!is_v) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float2 c = cs[static_cast<size_t>(half * 32 + j) * e.max_pos];
          const float x1 = a[j], x2 = b[j];
          a[j] = x1 * c.x - x2 * c.y;
          b[j] = x2 * c.x + x1 * c.y;
        }
      }
      uint4* o1 = reinterpret_cast<uint4*>(out + half * 32);
      uint4* o2 = reinterpret_cast<uint4*>(out + 64 + half * 32);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        o1[j] = make_uint4(pack2(a[8 * j], a[8 * j + 1]), pack2(a[8 * j + 2], a[8 * j + 3]), pack2(a[8 * j + 4], a[8 * j + 5]),
                           pack2(a[8 * j + 6], a[8 * j + 7]));
        o2[j] = make_uint4(pack2(b[8 * j], b[8 * j + 1]), pack2(b[8 * j + 2], b[8 * j + 3]), pack2(b[8 * j + 4], b[8 * j + 5]),
                           pack2(b[8 * j + 6], b[8 * j + 7]));
      }
      if (out_lo) {  // value - fp16(value), itself rounded to fp16
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          a[j] -= a2f(f2a(a[j]));
          b[j] -= a2f(f2a(b[j]));
        }
        uint4* l1 = reinterpret_cast<uint4*>(out_lo + half * 32);
        uint4* l2 = reinterpret_cast<uint4*>(out_lo + 64 + half * 32);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          l1[j] = make_uint4(pack2(a[8 * j], a[8 * j + 1]), pack2(a[8 * j + 2], a[8 * j + 3]),
                             pack2(a[8 * j + 4], a[8 * j + 5]), pack2(a[8 * j + 6], a[8 * j + 7]));
          l2[j] = make_uint4(pack2(b[8 * j], b[8 * j + 1]), pack2(b[8 * j + 2], b[8 * j + 3]),
                             pack2(b[8 * j + 4], b[8 * j + 5]), pack2(b[8 * j + 6], b[8 * j + 7]));
        }
      }
    }
  }
}

// ALO: A is given as two fp16 matrices, hi and lo (hi + lo carries ~22 bits of
// the activation); both are multiplied by the same B tile into one
// accumulator, so the weights are read once.
template <int MT, int BN, int EPI, bool ALO>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                   const GemmParams p, const EpiArgs e) {
  using C = GemmCfg<MT, BN, ALO>;
  // narrow tail units (tmB2: 64-row B boxes) exist only for single-tile CTAs
  // with an elementwise epilogue
  constexpr int NW = 64;
  constexpr bool kTail = MT == 1 && EPI == EPI_SWIGLU && BN > NW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + C::ACC_STAGES;
  uint64_t* drain = tempty + C::ACC_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // work distribution: CTA b takes units b, b + gridDim.x, ...
  const int slot = static_cast<int>(blockIdx.x);
  const int stride = static_cast<int>(gridDim.x);
  const int mtiles = (p.M + 127) / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < C::ACC_STAGES; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (ALO) tma_prefetch_desc(&tmA2);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tmem_slot;

  // unit u: its N tile (full width) or -1, M group, K split, first column and width
  auto unit = [&](int u, int& nt, int& mg, int& ks, int& col0, int& width) {
    if (!kTail || u < p.n_wide) {
      decode_unit(p, u, nt, mg, ks);
      col0 = nt * BN;
      width = BN;
    } else {
      const int v = u - p.n_wide;
      mg = v % p.n_mgroups;
      ks = 0;
      nt = -1;
      col0 = p.nw_col0 + (v / p.n_mgroups) * NW;
      width = NW;
    }
  };
  auto tile0 = [&](int mg) { return mg * MT; };  // this CTA's first M tile of group mg
  auto valid_tiles = [&](int mg) { return max(0, min(MT, mtiles - tile0(mg))); };
  // bytes one stage of unit (mg) receives: its A tiles (and lo halves), then B
  auto stage_bytes = [&](int mg, int width) {
    const int mt_valid = valid_tiles(mg);
    int lo_tiles = 0;
    if constexpr (ALO)
      for (int mt = 0; mt < mt_valid; ++mt) lo_tiles += ((tile0(mg) + mt + 1) * 128 > p.lo_row0) ? 1 : 0;
    return static_cast<uint32_t>((mt_valid + lo_tiles) * C::A_BYTES + width * 128);
  };
  const uint64_t pol_b = p.b_evict_first ? l2_policy_evict_first() : l2_policy_evict_last();
  auto load_b = [&](int stage, int kb, int col0, int width) {
    uint8_t* bdst = smem + stage * C::STAGE_BYTES + C::A_PARTS * MT * C::A_BYTES;
    tma_load_2d_hint(bdst, (kTail && width != BN) ? &tmB2 : &tmB, &full[stage], kb * 64, col0, pol_b);
  };
  // The weights do not depend on the previous kernel: the first STAGES
  // stages (all empty now) get their B tiles before the wait below, in the
  // producer's own (unit, k block) order; their A tiles follow after it.
  int pre = 0;
  uint32_t a_owed[8];  // A bytes a prologue stage still expects (its A loads not yet issued)
  for (int s = 0; s < 8; ++s) a_owed[s] = 0;
  if (p.b_const && warp == 0 && lane == 0) {
    for (int u = slot; u < p.n_units && pre < C::STAGES; u += stride) {
      int nt, mg, ks, col0, width;
      unit(u, nt, mg, ks, col0, width);
      const int kb0 = ks * p.nkb / p.k_splits, kb1 = (ks + 1) * p.nkb / p.k_splits;
      const uint32_t bytes = stage_bytes(mg, width);
      for (int kb = kb0; kb < kb1 && pre < C::STAGES; ++kb, ++pre) {
        mbar_arrive_expect_tx(&full[pre], bytes);
        load_b(pre, kb, col0, width);
        a_owed[pre] = bytes - static_cast<uint32_t>(width) * 128u;
      }
    }
  }
  // the prologue above overlapped the previous kernel's tail; its results are needed from here on
  griddep_launch_dependents();
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0, it = 0;
      uint32_t phase = 0;
      uint32_t last_phase[8];
      bool issued[8];
      for (int s = 0; s < 8; ++s) issued[s] = s < pre, last_phase[s] = 0;
      for (int u = slot; u < p.n_units && !*abort_flag; u += stride) {
        int nt, mg, ks, col0, width;
        unit(u, nt, mg, ks, col0, width);
        const int kb0 = ks * p.nkb / p.k_splits, kb1 = (ks + 1) * p.nkb / p.k_splits;
        const int mt_valid = valid_tiles(mg);
        const uint32_t bytes = stage_bytes(mg, width);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const bool b_done = it < pre;  // B already issued before the wait (first use of the stage)
          if (!b_done) {
            if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns)) {
              record_error(p.err, DEV_WAIT_TIMEOUT_PRODUCER);
              *abort_flag = 1;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], bytes);
          }
          uint8_t* base = smem + stage * C::STAGE_BYTES;
          for (int mt = 0; mt < mt_valid; ++mt) {
            tma_load_2d(base + mt * C::A_BYTES, &tmA, &full[stage], kb * 64, (tile0(mg) + mt) * 128);
            if constexpr (ALO)
              if ((tile0(mg) + mt + 1) * 128 > p.lo_row0)
                tma_load_2d(base + (MT + mt) * C::A_BYTES, &tmA2, &full[stage], kb * 64, (tile0(mg) + mt) * 128);
          }
          if (!b_done) load_b(stage, kb, col0, width);
          a_owed[stage] = 0;
          issued[stage] = true;
          last_phase[stage] = phase;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // let every copy still in flight land before the CTA exits: another warp
      // may have given up after this loop issued its last load (in a normal
      // run these phases are complete and the waits return at once)
      // (a prologue stage left without its A tiles by an abort is owed their
      // bytes, so that its phase completes once its B tile has landed)
      for (int s = 0; s < C::STAGES; ++s) {
        if (a_owed[s]) mbar_complete_tx(&full[s], a_owed[s]);
        if (issued[s]) mbar_wait(&full[s], last_phase[s], kDrainWaitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_W = idesc_f16_f32(128, BN);
      constexpr uint32_t IDESC_N = idesc_f16_f32(128, NW);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool any = false;
      for (int u = slot; u < p.n_units && !*abort_flag; u += stride) {
        int nt, mg, ks, col0, width;
        unit(u, nt, mg, ks, col0, width);
        const uint32_t IDESC = (kTail && width != BN) ? IDESC_N : IDESC_W;
        const int kb0 = ks * p.nkb / p.k_splits, kb1 = (ks + 1) * p.nkb / p.k_splits;
        const int mt_valid = valid_tiles(mg);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, p.wait_ns)) {
          record_error(p.err, DEV_WAIT_TIMEOUT_MMA);
          *abort_flag = 1;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_base = tbase + acc * C::ACC_COLS;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.wait_ns)) {
            record_error(p.err, DEV_WAIT_TIMEOUT_MMA);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_base = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b_base = a_base + C::A_PARTS * MT * C::A_BYTES;
          for (int mt = 0; mt < mt_valid; ++mt) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              umma_f16(d_base + mt * BN, sdesc_kmajor_sw128(a_base + mt * C::A_BYTES + k * 32),
                       sdesc_kmajor_sw128(b_base + k * 32), IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
            }
            if constexpr (ALO) {
              if ((tile0(mg) + mt + 1) * 128 > p.lo_row0)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                umma_f16(d_base + mt * BN, sdesc_kmajor_sw128(a_base + (MT + mt) * C::A_BYTES + k * 32),
                         sdesc_kmajor_sw128(b_base + k * 32), IDESC, 1u);
            }
          }
          umma_commit(&empty[stage]);
          any = true;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == C::ACC_STAGES) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // every MMA must be finished before TMEM is released
      if (any) {
        umma_commit(drain);
        if (!mbar_wait(drain, 0, kDrainWaitNs)) record_error(p.err, DEV_WAIT_TIMEOUT_DRAIN);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = slot; u < p.n_units && !*abort_flag; u += stride) {
      int nt, mg, ks, ucol0, width;
      unit(u, nt, mg, ks, ucol0, width);
      const int mt_valid = valid_tiles(mg);
      if (!mbar_wait(&tfull[acc], acc_phase, p.wait_ns)) {
        record_error(p.err, DEV_WAIT_TIMEOUT_EPILOGUE);
        *abort_flag = 1;
        break;
      }
      tc_fence_after_sync();
      for (int mt = 0; mt < mt_valid; ++mt) {
        const int tile = tile0(mg) + mt;
        const int row = tile * 128 + q * 32 + lane;
        const uint32_t t_row = tbase + (static_cast<uint32_t>(q * 32) << 16) + acc * C::ACC_COLS + mt * BN;
        float run_m = -INFINITY, run_s = 0.f;
        if constexpr (EPI == EPI_QKV_ROPE) {
          epi_qkv_rope<BN>(p, e, row, nt, t_row);
        } else {
          for (int c = 0; c < width / 32; ++c) {
            const int col0 = ucol0 + c * 32;
            if (col0 >= p.N) break;  // uniform across the warp
            float v[32];
            tmem_ld_32cols(t_row + c * 32, v);
            epi_chunk<EPI>(p, e, row, col0, v, run_m, run_s);
          }
        }
        if constexpr (EPI == EPI_READOUT) {
          if (row < p.M) e.part[static_cast<size_t>(nt) * p.M + row] = make_float2(run_m, run_s);
          // gathered logits: entries are sorted by N tile; the loop is uniform per warp
          const int g0 = e.gather_off[nt], g1 = e.gather_off[nt + 1];
          for (int g = g0; g < g1; ++g) {
            const int4 en = e.gather[g];
            const int r = en.y;
            if (r / 128 != tile || ((r & 127) >> 5) != q) continue;
            const float z = tmem_ld_1col(t_row + en.x);
            if (lane == (r & 31)) e.z_out[en.z] = z;
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&tempty[acc]);
      if (++acc == C::ACC_STAGES) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

// ====================================================================== CTA pairs
// The same GEMM on a pair of CTAs (a 2-CTA cluster) sharing one tcgen05 MMA of
// M = 256: each CTA loads its own 128 rows of A and half of the B tile (BN/2
// rows), so a k block brings 16 KB of A + BN/2 x 128 B of B into each SM
// instead of 16 KB + BN x 128 B — the fill of each SM's shared memory is what
// bounds the single-CTA mainloop at these sizes.  The leader (rank 0) issues
// the MMAs; both CTAs run the epilogue on their own accumulator rows.
template <int BN, bool ALO>
struct PairCfg {
  static constexpr int A_BYTES = 128 * 128;        // 128 rows x 64 fp16
  static constexpr int B_BYTES = (BN / 2) * 128;   // this CTA's half of the B tile
  static constexpr int A_PARTS = ALO ? 2 : 1;
  static constexpr int STAGE_BYTES = A_PARTS * A_BYTES + B_BYTES;
  static constexpr int SMEM_BUDGET = 227 * 1024 - 2048;
  static constexpr int STAGES_RAW = SMEM_BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
  static constexpr int ACC_COLS = BN;
  static constexpr int ACC_STAGES = (2 * ACC_COLS <= 512) ? 2 : 1;
  static constexpr int TMEM_RAW = ACC_STAGES * ACC_COLS;
  static constexpr int TMEM_COLS = TMEM_RAW <= 32 ? 32 : TMEM_RAW <= 64 ? 64 : TMEM_RAW <= 128 ? 128 : TMEM_RAW <= 256 ? 256 : 512;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 512;
  static_assert(STAGES >= 2, "at least two stages");
  static_assert((2 * STAGES + 2 * ACC_STAGES + 1) * 8 + 8 + 8 * STAGES <= 512, "barriers and drain counts fit");
};

template <int BN, int EPI, bool ALO>
__global__ void __launch_bounds__(192, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmA2, const GemmParams p, const EpiArgs e) {
  using C = PairCfg<BN, ALO>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);  // used in the leader
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + C::ACC_STAGES;  // used in the leader
  uint64_t* drain = tempty + C::ACC_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());  // 0: leader
  const int pair = static_cast<int>(cluster_id_x());
  const int n_pairs = static_cast<int>(n_clusters_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);  // the leader's producer expects both CTAs' bytes
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < C::ACC_STAGES; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 256);  // every epilogue thread of both CTAs
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (ALO) tma_prefetch_desc(&tmA2);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync_all();  // the leader's barriers exist before the peer signals them
  tc_fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  griddep_launch_dependents();
  griddep_wait();

  auto row0 = [&](int mg) { return mg * 256 + rank * 128; };  // this CTA's first row of pair tile mg
  // a pair tile carries the A remainder when any of its rows is at or past lo_row0 (both CTAs alike)
  auto has_lo = [&](int mg) { return ALO && (mg + 1) * 256 > p.lo_row0; };

  // phases this CTA's producer issued into each stage and the bytes of the
  // last one; the peer reports its counts to the leader, which completes the
  // drain (see the end of the kernel)
  uint32_t* peer_cnt = tmem_slot + 2;  // [C::STAGES], after the TMEM slot and the abort flag
  uint32_t* peer_last = peer_cnt + C::STAGES;
  uint32_t cnt[C::STAGES], last[C::STAGES];
  for (int s2 = 0; s2 < C::STAGES; ++s2) cnt[s2] = 0, last[s2] = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int u = pair; u < p.n_units && !*abort_flag; u += n_pairs) {
        int nt, mg, ks;
        decode_unit(p, u, nt, mg, ks);
        const int kb0 = ks * p.nkb / p.k_splits, kb1 = (ks + 1) * p.nkb / p.k_splits;
        const bool lo = has_lo(mg);
        const uint32_t bytes = (lo ? 2 : 1) * C::A_BYTES + C::B_BYTES;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_ns)) {
            record_error(p.err, DEV_WAIT_TIMEOUT_PRODUCER);
            *abort_flag = 1;
            break;
          }
          // the stage's bytes from both CTAs complete the leader's barrier; only
          // the leader arrives on it (a remote arrive per stage from the peer
          // measured twice as slow)
          const uint32_t fb = cluster_addr(&full[stage], 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * bytes);
          uint8_t* base = smem + stage * C::STAGE_BYTES;
          tma_load_2d_pair(base, &tmA, fb, kb * 64, row0(mg));
          if constexpr (ALO)
            if (lo) tma_load_2d_pair(base + C::A_BYTES, &tmA2, fb, kb * 64, row0(mg));
          tma_load_2d_pair(base + C::A_PARTS * C::A_BYTES, &tmB, fb, kb * 64, nt * BN + rank * (BN / 2));
          cnt[stage] += 1;
          last[stage] = bytes;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (rank == 1)
        for (int s2 = 0; s2 < C::STAGES; ++s2) {
          asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr(&peer_cnt[s2], 0)), "r"(cnt[s2]) : "memory");
          asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr(&peer_last[s2], 0)), "r"(last[s2])
                       : "memory");
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t IDESC = idesc_f16_f32(256, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool any = false;
      for (int u = pair; u < p.n_units && !*abort_flag; u += n_pairs) {
        int nt, mg, ks;
        decode_unit(p, u, nt, mg, ks);
        const int kb0 = ks * p.nkb / p.k_splits, kb1 = (ks + 1) * p.nkb / p.k_splits;
        const bool lo = has_lo(mg);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, p.wait_ns)) {
          record_error(p.err, DEV_WAIT_TIMEOUT_MMA);
          *abort_flag = 1;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_base = tbase + acc * C::ACC_COLS;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.wait_ns)) {
            record_error(p.err, DEV_WAIT_TIMEOUT_MMA);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_base = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b_base = a_base + C::A_PARTS * C::A_BYTES;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_f16_pair(d_base, sdesc_kmajor_sw128(a_base + k * 32), sdesc_kmajor_sw128(b_base + k * 32), IDESC,
                          (kb > kb0 || k > 0) ? 1u : 0u);
          if constexpr (ALO)
            if (lo)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                umma_f16_pair(d_base, sdesc_kmajor_sw128(a_base + C::A_BYTES + k * 32),
                              sdesc_kmajor_sw128(b_base + k * 32), IDESC, 1u);
          umma_commit_pair_mc(&empty[stage]);  // both CTAs' stage is free once these MMAs are done
          any = true;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(&tfull[acc]);
        if (++acc == C::ACC_STAGES) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (any) {
        umma_commit_pair(drain);
        if (!mbar_wait(drain, 0, kDrainWaitNs)) record_error(p.err, DEV_WAIT_TIMEOUT_DRAIN);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = pair; u < p.n_units && !*abort_flag; u += n_pairs) {
      int nt, mg, ks;
      decode_unit(p, u, nt, mg, ks);
      if (!mbar_wait(&tfull[acc], acc_phase, p.wait_ns)) {
        record_error(p.err, DEV_WAIT_TIMEOUT_EPILOGUE);
        *abort_flag = 1;
        break;
      }
      tc_fence_after_sync();
      const int tile = mg * 2 + rank;  // this CTA's 128-row tile
      const int row = tile * 128 + q * 32 + lane;
      const uint32_t t_row = tbase + (static_cast<uint32_t>(q * 32) << 16) + acc * C::ACC_COLS;
      float run_m = -INFINITY, run_s = 0.f;
      if constexpr (EPI == EPI_QKV_ROPE) {
        epi_qkv_rope<BN>(p, e, row, nt, t_row);
      } else {
        for (int c = 0; c < BN / 32; ++c) {
          const int col0 = nt * BN + c * 32;
          if (col0 >= p.N) break;  // uniform across the warp
          float v[32];
          tmem_ld_32cols(t_row + c * 32, v);
          epi_chunk<EPI>(p, e, row, col0, v, run_m, run_s);
        }
      }
      if constexpr (EPI == EPI_READOUT) {
        if (row < p.M) e.part[static_cast<size_t>(nt) * p.M + row] = make_float2(run_m, run_s);
        const int g0 = e.gather_off[nt], g1 = e.gather_off[nt + 1];
        for (int g = g0; g < g1; ++g) {
          const int4 en = e.gather[g];
          const int r = en.y;
          if (r / 128 != tile || ((r & 127) >> 5) != q) continue;
          const float z = tmem_ld_1col(t_row + en.x);
          if (lane == (r & 31)) e.z_out[en.z] = z;
        }
      }
      tc_fence_before_sync();
      mbar_arrive_cluster(cluster_addr(&tempty[acc], 0));  // the leader may reuse the accumulator
      if (++acc == C::ACC_STAGES) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before_sync();
  cluster_sync_all();  // no copy is issued after this; the peer's counts are visible to the leader
  if (warp == 0 && lane == 0 && rank == 0) {
    // every phase either CTA issued into completes before either exits: a
    // phase this CTA armed that the peer never loaded is owed the peer's bytes;
    // one the peer loaded ahead of this CTA's arming is armed with them (each
    // CTA's ring waits on the previous phase of the other, so the counts
    // differ by at most one)
    for (int s2 = 0; s2 < C::STAGES; ++s2) {
      const uint32_t a = cnt[s2], n = peer_cnt[s2], pb = peer_last[s2];
      if (a == 0 && n == 0) continue;
      if (n > a + 1 || n + 1 < a) {
        record_error(p.err, DEV_WAIT_TIMEOUT_DRAIN);
        continue;
      }
      uint32_t ph;
      if (n == a + 1) {
        mbar_arrive_expect_tx(&full[s2], pb);
        ph = n - 1;
      } else {
        if (n + 1 == a) mbar_complete_tx(&full[s2], last[s2]);
        ph = a - 1;
      }
      if (!mbar_wait(&full[s2], ph & 1u, kDrainWaitNs)) record_error(p.err, DEV_WAIT_TIMEOUT_DRAIN);
    }
  }
  tc_fence_before_sync();
  cluster_sync_all();  // neither CTA's shared memory or barriers are touched by the other after this
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tbase, C::TMEM_COLS);
  }
}

// ====================================================================== host
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

bool tma_init() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 16-bit matrix [rows][>= cols], row stride ld elements; box 64 (K) x box_rows.
// Encoded maps are cached by (pointer, shape, box): the executor reuses the
// same weight and workspace matrices every call.
struct MapKey {
  uintptr_t p;
  int rows, cols, ld, box;
  bool operator==(const MapKey& o) const {
    return p == o.p && rows == o.rows && cols == o.cols && ld == o.ld && box == o.box;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    size_t h = std::hash<uintptr_t>()(k.p);
    for (int v : {k.rows, k.cols, k.ld, k.box}) h = h * 1000003u ^ static_cast<size_t>(v);
    return h;
  }
};
static std::mutex g_map_mu;
static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

static bool encode_map(CUtensorMap* m, const void* ptr, int rows, int cols, int ld, int box_rows);

static bool make_map(CUtensorMap* m, const void* ptr, int rows, int cols, int ld, int box_rows) {
  const MapKey k{reinterpret_cast<uintptr_t>(ptr), rows, cols, ld, box_rows};
  std::lock_guard<std::mutex> lock(g_map_mu);
  auto it = g_maps.find(k);
  if (it != g_maps.end()) {
    *m = it->second;
    return true;
  }
  if (!encode_map(m, ptr, rows, cols, ld, box_rows)) return false;
  if (g_maps.size() > 4096) g_maps.clear();
  g_maps.emplace(k, *m);
  return true;
}

bool make_tile_map(CUtensorMap* m, const void* ptr, int rows, int cols, int ld, int box_rows) {
  return make_map(m, ptr, rows, cols, ld, box_rows);
}

static bool encode_map(CUtensorMap* m, const void* ptr, int rows, int cols, int ld, int box_rows) {
  if (!tma_init()) return false;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || (ld * 2) % 16) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_kv_map(CUtensorMap* m, const void* base, int dh, int n_rows, int n_heads, int64_t head_rows, int n_layers,
                 int64_t layer_elems) {
  static std::mutex mu;
  static std::map<std::tuple<uintptr_t, int, int, int, int64_t, int, int64_t>, CUtensorMap> cache;
  const auto key = std::make_tuple(reinterpret_cast<uintptr_t>(base), dh, n_rows, n_heads, head_rows, n_layers,
                                   layer_elems);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *m = it->second;
    return true;
  }
  if (!tma_init() || n_rows < 1 || dh % 64 || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(dh), static_cast<cuuint64_t>(n_rows), static_cast<cuuint64_t>(n_heads),
                        static_cast<cuuint64_t>(n_layers)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(dh) * 2, static_cast<cuuint64_t>(head_rows) * dh * 2,
                           static_cast<cuuint64_t>(layer_elems) * 2};
  cuuint32_t box[4] = {64, 64, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (cache.size() > 1024) cache.clear();
  cache.emplace(key, *m);
  return true;
}

bool make_q_map(CUtensorMap* m, const void* base, int dh, int n_heads, int n_rows, int box_heads, int box_rows) {
  static std::mutex mu;
  static std::map<std::tuple<uintptr_t, int, int, int, int, int>, CUtensorMap> cache;
  const auto key = std::make_tuple(reinterpret_cast<uintptr_t>(base), dh, n_heads, n_rows, box_heads, box_rows);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *m = it->second;
    return true;
  }
  if (!tma_init() || n_rows < 1 || dh % 64 || box_heads < 1 || box_heads > 256 || box_rows < 1 || box_rows > 256 ||
      (reinterpret_cast<uintptr_t>(base) & 15))
    return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(dh), static_cast<cuuint64_t>(n_heads), static_cast<cuuint64_t>(n_rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(dh) * 2, static_cast<cuuint64_t>(n_heads) * dh * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_heads), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (cache.size() > 1024) cache.clear();
  cache.emplace(key, *m);
  return true;
}

template <int MT, int BN, int EPI, bool ALO = false>
static int launch_t(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& ma2, const CUtensorMap& mb2,
                    const GemmParams& p, const EpiArgs& e, cudaStream_t st, int sms) {
  using C = GemmCfg<MT, BN, ALO>;
  auto kern = gemm_tc_kernel<MT, BN, EPI, ALO>;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (r != cudaSuccess) return r;
    attr_set = true;
  }
  const int grid = std::min(p.n_units, sms);
  return launch_k(kern, dim3(grid), dim3(192), C::SMEM_BYTES, st, ma, mb, ma2, mb2, p, e);
}

template <int BN, int EPI, bool ALO>
static int launch_pair(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& ma2, const GemmParams& p,
                       const EpiArgs& e, cudaStream_t st, int sms) {
  using C = PairCfg<BN, ALO>;
  auto kern = gemm_pair_kernel<BN, EPI, ALO>;
  static bool attr_set = false;  // per instantiation
  static int max_pairs = 0;
  if (!attr_set) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (r != cudaSuccess) return r;
    // how many pairs can be resident at once: the kernel is persistent
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(2 * (sms / 2), 1, 1);
    q.blockDim = dim3(192, 1, 1);
    q.dynamicSmemBytes = C::SMEM_BYTES;
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
    attr_set = true;
  }
  const int pairs = std::min(p.n_units, max_pairs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, ma, mb, ma2, p, e);
}

template <int EPI>
static int dispatch_tiling(const GemmTiling& t, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap* ma2,
                           const CUtensorMap& mb2, const GemmParams& p, const EpiArgs& e, cudaStream_t st, int sms) {
  if (t.pair) {
    if (ma2) {
      if (t.bn == 128) return launch_pair<128, EPI, true>(ma, mb, *ma2, p, e, st, sms);
      if (t.bn == 256) return launch_pair<256, EPI, true>(ma, mb, *ma2, p, e, st, sms);
    } else {
      if (t.bn == 128) return launch_pair<128, EPI, false>(ma, mb, ma, p, e, st, sms);
      if (t.bn == 256) return launch_pair<256, EPI, false>(ma, mb, ma, p, e, st, sms);
    }
    return -1;
  }
  if (ma2) {  // hi + lo A: one 128-row tile per CTA
    if constexpr (EPI == EPI_F32_STORE || EPI == EPI_F32_ADD || EPI == EPI_F32_ATOMIC || EPI == EPI_SWIGLU ||
                  EPI == EPI_READOUT || EPI == EPI_QKV_ROPE) {
      if (t.mt == 1 && t.bn == 128) return launch_t<1, 128, EPI, true>(ma, mb, *ma2, mb2, p, e, st, sms);
      if (t.mt == 1 && t.bn == 256) return launch_t<1, 256, EPI, true>(ma, mb, *ma2, mb2, p, e, st, sms);
    }
    return -1;
  }
  if (t.mt == 1 && t.bn == 128) return launch_t<1, 128, EPI>(ma, mb, ma, mb2, p, e, st, sms);
  if (t.mt == 1 && t.bn == 256) return launch_t<1, 256, EPI>(ma, mb, ma, mb2, p, e, st, sms);
  if (t.mt == 2 && t.bn == 128) return launch_t<2, 128, EPI>(ma, mb, ma, mb2, p, e, st, sms);
  if (t.mt == 2 && t.bn == 256) return launch_t<2, 256, EPI>(ma, mb, ma, mb2, p, e, st, sms);
  if (t.mt == 4 && t.bn == 128) return launch_t<4, 128, EPI>(ma, mb, ma, mb2, p, e, st, sms);
  return -1;
}

int launch_gemm(const GemmShape& s, int epi, const EpiArgs& e, const GemmTiling& t, cudaStream_t stream, int* dev_err,
                uint64_t wait_ns, int sms) {
  const int M = s.a_rows, N = s.b_rows, K = s.K;
  if (M <= 0 || N <= 0) return 0;
  if (K <= 0 || K % 64 || N % 32) return -1;
  if (t.splits > 1 && epi != EPI_F32_ATOMIC) return -1;
  GemmParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.nkb = K / 64;
  if (t.pair && t.mt != 1) return -1;
  p.n_mgroups = ceil_div(M, t.pair ? 256 : 128 * t.mt);
  p.n_ntiles = ceil_div(N, t.bn);
  p.k_splits = std::max(1, std::min(t.splits, p.nkb));
  p.n_units = p.n_mgroups * p.n_ntiles * p.k_splits;
  p.wait_ns = wait_ns;
  p.err = dev_err;
  p.b_evict_first = (p.n_mgroups == 1 && (t.pair ? 256 : t.mt * 128) >= M) ? 1 : 0;
  p.lo_row0 = s.lo_row0;
  p.b_const = s.b_const ? 1 : 0;
  // the last wave's tail: when the units leave the final wave part-filled,
  // the last N tiles run as 64-column units instead, filling that wave with
  // shorter work (elementwise SwiGLU epilogue, single-tile CTAs)
  p.n_wide = p.n_units;
  p.nw_col0 = 0;
  static const bool tail_on = [] {
    const char* v = std::getenv("PCD_GEMM_TAIL");
    return !v || std::atoi(v) != 0;
  }();
  if (tail_on && epi == EPI_SWIGLU && t.mt == 1 && !t.pair && p.k_splits == 1 && t.bn > 64 &&
      N % t.bn == 0) {
    const int grid = std::min(p.n_units, sms);
    const int waves = p.n_units / grid, rest = p.n_units - waves * grid;
    if (waves >= 1 && rest > 0) {
      const int tt = ceil_div(rest, p.n_mgroups);  // N tiles turned into 64-column units
      const int narrow = tt * (t.bn / 64) * p.n_mgroups;
      if (tt < p.n_ntiles && narrow <= grid) {
        p.n_wide = (p.n_ntiles - tt) * p.n_mgroups;
        p.nw_col0 = (p.n_ntiles - tt) * t.bn;
        p.n_units = p.n_wide + narrow;
      }
    }
  }
  CUtensorMap ma, mb, ma2, mb2;
  if (!make_map(&ma, s.a, M, K, s.a_ld, 128)) return -1;
  if (s.a_lo && !make_map(&ma2, s.a_lo, M, K, s.a_ld, 128)) return -1;
  const CUtensorMap* pa2 = s.a_lo ? &ma2 : nullptr;
  if (!make_map(&mb, s.b, N, K, s.b_ld, t.pair ? t.bn / 2 : t.bn)) return -1;
  if (p.n_wide < p.n_units) {
    if (!make_map(&mb2, s.b, N, K, s.b_ld, 64)) return -1;
  } else {
    mb2 = mb;
  }
  switch (epi) {
    case EPI_BF16: return dispatch_tiling<EPI_BF16>(t, ma, mb, pa2, mb2, p, e, stream, sms);
    case EPI_F32_ADD: return dispatch_tiling<EPI_F32_ADD>(t, ma, mb, pa2, mb2, p, e, stream, sms);
    case EPI_F32_ATOMIC: return dispatch_tiling<EPI_F32_ATOMIC>(t, ma, mb, pa2, mb2, p, e, stream, sms);
    case EPI_SWIGLU: return dispatch_tiling<EPI_SWIGLU>(t, ma, mb, pa2, mb2, p, e, stream, sms);
    case EPI_READOUT: return dispatch_tiling<EPI_READOUT>(t, ma, mb, pa2, mb2, p, e, stream, sms);
    case EPI_F32_STORE: return dispatch_tiling<EPI_F32_STORE>(t, ma, mb, pa2, mb2, p, e, stream, sms);
    case EPI_QKV_ROPE:
      if (t.splits != 1 || t.bn % 128 || N % 128) return -1;
      return dispatch_tiling<EPI_QKV_ROPE>(t, ma, mb, pa2, mb2, p, e, stream, sms);
  }
  return -1;
}

// Tiling heuristic (calibrated on GB300).  One 128-row M tile per work unit:
// it leaves room for the deepest stage ring, and the units that share a B
// tile run on neighbouring CTAs and share it through L2.  A k-block costs the
// larger of its MMA time (128 x BN x 64 x 2 flop at ~8192 flop/clk/SM) and its
// shared-memory fill ((128 + BN) x 128 bytes at ~60 B/clk/SM, the rate a
// 128x256 tile sustains at 82% of peak); a unit adds a fixed pipeline fill and
// epilogue cost; waves of `sms` units run back to back.
GemmTiling choose_tiling(int M, int N, int K, int epi, int sms) {
  const int nkb = K / 64;
  const int mtiles = ceil_div(M, 128);
  GemmTiling best;
  best.mt = 1;
  double best_t = 1e30;
  for (int bn : {128, 256}) {
    const int nt = ceil_div(N, bn);
    const int max_split = (epi == EPI_F32_ATOMIC) ? std::max(1, std::min(16, nkb / 3)) : 1;
    for (int sp = 1; sp <= max_split; ++sp) {
      const int units = mtiles * nt * sp;
      const int kbs = ceil_div(nkb, sp);
      // cycles per 64-deep k block: the MMA, or filling shared memory with
      // the A and B tiles at ~55 B/clk per SM (measured with every SM loading)
      const double mma = 128.0 * bn * 128.0 / 8192.0;
      const double fill = (128.0 + bn) * 128.0 / 55.0;
      // a unit's fixed cost: pipeline ramp, plus the fp32 atomics of a split-K epilogue
      const double fixed = (epi == EPI_F32_ATOMIC) ? 7000.0 : 2500.0;
      const double per_unit = kbs * std::max(mma, fill) + fixed;
      const double tt = ceil_div(units, std::max(1, sms)) * per_unit + (sp > 1 ? 400.0 : 0.0);
      if (tt < best_t * 0.97) {
        best_t = tt;
        best.bn = bn;
        best.splits = sp;
        best.pair = false;
      }
    }
  }
  // Short SwiGLU projections (the branch and single-pass row counts): two
  // 128-row tiles per unit share each 256-column B tile, which halves the
  // units (one wave instead of two at 313 rows: 21.8 vs 24.6 us for the
  // 1.5B gate/up; 38.8 vs 39.9 us at 825 rows).  At thousands of rows the
  // single accumulator stage and three-deep ring of this form lose (467 vs
  // 282 us at 8192 rows), so it stays below 1024 rows.
  if (epi == EPI_SWIGLU && M > 128 && M <= 1024 && N % 256 == 0) {
    best.mt = 2;
    best.bn = 256;
    best.splits = 1;
    best.pair = false;
    return best;
  }
  // CTA pairs: 256-row tiles on two SMs, each SM filling its 128 A rows and
  // half of the B tile per k block (off unless PCD_GEMM_PAIR allows them)
  static const bool allow_pair = [] {
    const char* e = std::getenv("PCD_GEMM_PAIR");
    return e && std::atoi(e) != 0;
  }();
  if (allow_pair) {
    const int pgroups = ceil_div(M, 256);
    for (int bn : {128, 256}) {
      const int nt = ceil_div(N, bn);
      const int max_split = (epi == EPI_F32_ATOMIC) ? std::max(1, std::min(16, nkb / 3)) : 1;
      for (int sp = 1; sp <= max_split; ++sp) {
        const int units = pgroups * nt * sp;
        const int slots = std::max(1, sms / 2);
        const int kbs = ceil_div(nkb, sp);
        const double mma = 128.0 * bn * 128.0 / 8192.0;
        const double fill = (128.0 + bn / 2) * 128.0 / 55.0;
        const double fixed = (epi == EPI_F32_ATOMIC) ? 7000.0 : 2500.0;
        const double tt = ceil_div(units, slots) * (kbs * std::max(mma, fill) + fixed) + (sp > 1 ? 400.0 : 0.0);
        if (tt < best_t * 0.97) {
          best_t = tt;
          best.bn = bn;
          best.splits = sp;
          best.pair = true;
        }
      }
    }
  }
  return best;
}

}  // namespace pcd
