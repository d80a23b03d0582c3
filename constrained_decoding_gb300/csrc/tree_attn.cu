// Tree attention over a packed pass: causal prefix queries and branch queries
// (whole prefix + own ancestors) in one launch, with no partial results in
// global memory.
//
// The branch mask is the one the parallel-decoding pages describe: every
// branch token attends to the shared prefix and to the earlier tokens of its
// own branch only, never to another field's tokens ("Constrained decoding"
// pages, shared-prefix KV cache and per-field branches).  Positions are those
// the branch compiler assigned; the keys carry them through RoPE already.
#include <climits>
#include <cstdint>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "warp_mma.cuh"

namespace pcd {

template <int DH>
struct TreeSmem {
  static constexpr int LDS = DH + 8;        // padded fp16 row: conflict-free ldmatrix
  static constexpr int TILE = 64 * LDS;     // elements of one 64-row tile
  static constexpr int RED_LD = DH + 4;     // fp32 partial-output row stride (16-byte aligned rows)
  static constexpr int Q_BYTES = TILE * 2;
  static constexpr int KV_BYTES = 4 * TILE * 2;  // K and V, double-buffered
  static constexpr int BYTES = Q_BYTES + KV_BYTES + 64 * 8 /* (m, l) per row */ + 64 * 8 /* token masks */;
  static_assert(64 * RED_LD * 4 <= KV_BYTES, "the partial output reuses the K/V buffers");
};

// Grid: x = (branch tiles + prefix tiles) * csk, y = KV heads; the csk CTAs of
// one (tile, head) form a cluster.  Branch tiles come first, then prefix tiles
// from the last (most keys) to the first.  A CTA runs 4 warps x 16 query rows
// and takes key blocks rank, rank + csk, ... of its tile: the prefix key
// blocks, then the tile's ancestor chunks.
template <int DH>
__global__ void __launch_bounds__(128) tree_attn_kernel(TreeAttnArgs a) {
  using S = TreeSmem<DH>;
  constexpr int LDS = S::LDS;
  constexpr int KS = DH / 16;  // k-steps over the head dim
  constexpr int ND = DH / 8;   // 8-wide output column blocks
  constexpr int QCH = DH / 8;  // 16-byte chunks per row
  extern __shared__ __align__(16) uint8_t tree_smem[];
  act_t* sQ = reinterpret_cast<act_t*>(tree_smem);
  act_t* sK = sQ + S::TILE;      // [2][64][LDS]
  act_t* sV = sK + 2 * S::TILE;  // [2][64][LDS]
  float* sRed = reinterpret_cast<float*>(sK);  // [64][RED_LD] once the key loop is done
  float2* sML = reinterpret_cast<float2*>(tree_smem + S::Q_BYTES + S::KV_BYTES);
  unsigned long long* sMask = reinterpret_cast<unsigned long long*>(sML + 64);

  griddep_launch_dependents();
  griddep_wait();
  const int csk = a.csk;
  const int item = blockIdx.x / csk;
  const int rank = blockIdx.x - item * csk;  // == %cluster_ctarank for a (csk, 1, 1) cluster
  const int hk = blockIdx.y;
  const int G = a.Hq / a.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tq = lane & 3;

  const bool branch = item < a.n_br_tiles;
  const int tile = branch ? item : a.n_pf_tiles - 1 - (item - a.n_br_tiles);
  // a branch tile's tokens come from the plan (tiles end at request boundaries)
  const int t0 = branch ? a.tile_tok[3 * tile] : tile * a.tpt;
  const int ntok = branch ? a.tile_tok[3 * tile + 1] : min(a.tpt, a.n_pf - t0);
  const int qrow0 = branch ? a.br_row0 + t0 : t0;  // q / out row of the tile's first token
  const int rows = ntok * G;
  const int pf_keys = branch ? a.n_keys : min(a.n_keys, a.pf_pos0 + t0 + ntok);
  const int nbp = (pf_keys + 63) / 64;
  const int ch0 = branch ? a.tile_chunk_off[tile] : 0;
  const int nb = nbp + (branch ? a.tile_chunk_off[tile + 1] - ch0 : 0);
  const int my_n = rank < nb ? (nb - 1 - rank) / csk + 1 : 0;

  for (int c = tid; c < 64 * QCH; c += 128) {
    const int rr = c / QCH, ch = c % QCH;
    const bool ok = rr < rows;
    const int t = qrow0 + (ok ? rr / G : 0), g = ok ? rr % G : 0;
    cp_async16(sQ + rr * LDS + ch * 8, a.q + (static_cast<size_t>(t) * a.Hq + hk * G + g) * DH + ch * 8, ok);
  }
  cp_async_commit();

  const act_t* kp = a.k + static_cast<size_t>(hk) * a.kv_head_stride * DH;
  const act_t* vp = a.v + static_cast<size_t>(hk) * a.kv_head_stride * DH;
  const act_t* kbp = a.kb + static_cast<size_t>(hk) * a.n_br * DH;
  const act_t* vbp = a.vb + static_cast<size_t>(hk) * a.n_br * DH;
  auto load_kv = [&](int b, int buf) {
    act_t* dk = sK + buf * S::TILE;
    act_t* dv = sV + buf * S::TILE;
    if (b < nbp) {
      const int j0 = b * 64;
      for (int c = tid; c < 64 * QCH; c += 128) {
        const int kr = c / QCH, ch = c % QCH;
        const int j = j0 + kr;
        const bool ok = j < pf_keys;
        const size_t off = static_cast<size_t>(ok ? j : 0) * DH + ch * 8;
        cp_async16(dk + kr * LDS + ch * 8, kp + off, ok);
        cp_async16(dv + kr * LDS + ch * 8, vp + off, ok);
      }
    } else {
      const int32_t* keys = a.tile_keys + static_cast<size_t>(ch0 + b - nbp) * 64;
      for (int c = tid; c < 64 * QCH; c += 128) {
        const int kr = c / QCH, ch = c % QCH;
        const int j = keys[kr];
        const bool ok = j >= 0 && j < a.n_br;
        const size_t off = static_cast<size_t>(ok ? j : 0) * DH + ch * 8;
        cp_async16(dk + kr * LDS + ch * 8, kbp + off, ok);
        cp_async16(dv + kr * LDS + ch * 8, vbp + off, ok);
      }
    }
    cp_async_commit();
  };
  if (my_n > 0) {
    load_kv(rank, 0);
    cp_async_wait<1>();
  } else {
    cp_async_wait<0>();
  }
  __syncthreads();
  uint32_t qf[KS][4];
#pragma unroll
  for (int kk = 0; kk < KS; ++kk)
    ldsm_x4(qf[kk], sQ + (warp * 16 + (lane & 15)) * LDS + kk * 16 + (lane >> 4) * 8);

  const int rlo = warp * 16 + gid, rhi = rlo + 8;
  // causal bound of prefix rows (branch rows see every prefix key)
  const int pos_lo = branch ? INT_MAX : a.pf_pos0 + t0 + rlo / G;
  const int pos_hi = branch ? INT_MAX : a.pf_pos0 + t0 + rhi / G;
  const int tlo = rlo / G, thi = rhi / G;  // token of the row within the tile (< 64)
  float o[ND][4];
#pragma unroll
  for (int i = 0; i < ND; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

  for (int i = 0; i < my_n; ++i) {
    const int b = rank + i * csk;
    const int buf = i & 1;
    if (i + 1 < my_n) {
      load_kv(b + csk, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    const bool local = b >= nbp;
    if (local && tid < ntok) sMask[tid] = a.tile_mask[static_cast<size_t>(ch0 + b - nbp) * a.tpt + tid];
    __syncthreads();
    const act_t* K = sK + buf * S::TILE;
    const act_t* V = sV + buf * S::TILE;

    float s[8][4];
#pragma unroll
    for (int x = 0; x < 8; ++x) s[x][0] = s[x][1] = s[x][2] = s[x][3] = 0.f;
#pragma unroll
    for (int nb2 = 0; nb2 < 4; ++nb2) {
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        uint32_t bb[4];
        ldsm_x4(bb, K + (nb2 * 16 + (lane >> 4) * 8 + (lane & 7)) * LDS + kk * 16 + ((lane >> 3) & 1) * 8);
        mma16816(s[2 * nb2], qf[kk], bb[0], bb[1]);
        mma16816(s[2 * nb2 + 1], qf[kk], bb[2], bb[3]);
      }
    }
    // scale, mask, online softmax (log2 units)
    unsigned long long mk_lo = 0ull, mk_hi = 0ull;
    if (local) {
      mk_lo = sMask[tlo];
      mk_hi = sMask[thi];
    }
    const int j0 = b * 64;
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int x = 0; x < 8; ++x) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int jj = x * 8 + tq * 2 + e;  // key within the block
        bool v_lo, v_hi;
        if (local) {
          v_lo = (mk_lo >> jj) & 1ull;
          v_hi = (mk_hi >> jj) & 1ull;
        } else {
          const int j = j0 + jj;
          v_lo = j < pf_keys && j <= pos_lo;
          v_hi = j < pf_keys && j <= pos_hi;
        }
        const float s0 = v_lo ? s[x][e] * a.scale_log2 : -INFINITY;
        const float s1 = v_hi ? s[x][2 + e] * a.scale_log2 : -INFINITY;
        s[x][e] = s0;
        s[x][2 + e] = s1;
        mx_lo = fmaxf(mx_lo, s0);
        mx_hi = fmaxf(mx_hi, s1);
      }
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, off));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, off));
    }
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float c_lo = (mn_lo == -INFINITY) ? 1.f : exp2f(m_lo - mn_lo);
    const float c_hi = (mn_hi == -INFINITY) ? 1.f : exp2f(m_hi - mn_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
    float rs_lo = 0.f, rs_hi = 0.f;
#pragma unroll
    for (int x = 0; x < 8; ++x) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float p0 = (mn_lo == -INFINITY) ? 0.f : exp2f(s[x][e] - mn_lo);
        const float p1 = (mn_hi == -INFINITY) ? 0.f : exp2f(s[x][2 + e] - mn_hi);
        s[x][e] = p0;
        s[x][2 + e] = p1;
        rs_lo += p0;
        rs_hi += p1;
      }
    }
    l_lo = l_lo * c_lo + rs_lo;
    l_hi = l_hi * c_hi + rs_hi;
#pragma unroll
    for (int x = 0; x < ND; ++x) {
      o[x][0] *= c_lo;
      o[x][1] *= c_lo;
      o[x][2] *= c_hi;
      o[x][3] *= c_hi;
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack2(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack2(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int nd2 = 0; nd2 < DH / 16; ++nd2) {
        uint32_t bb[4];
        ldsm_x4_t(bb, V + (kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7)) * LDS + nd2 * 16 + (lane >> 4) * 8);
        mma16816(o[2 * nd2], pa, bb[0], bb[1]);
        mma16816(o[2 * nd2 + 1], pa, bb[2], bb[3]);
      }
    }
    __syncthreads();  // the buffer is refilled next iteration
  }

#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, off);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, off);
  }

  if (csk == 1) {
    const float il_lo = l_lo > 0.f ? 1.f / l_lo : 0.f;
    const float il_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = half ? rhi : rlo;
      if (r >= rows) continue;
      const float il = half ? il_hi : il_lo;
      const size_t base = static_cast<size_t>(qrow0 + r / G) * a.ld_out + (hk * G + r % G) * DH;
#pragma unroll
      for (int nd = 0; nd < ND; ++nd) {
        const int d = nd * 8 + tq * 2;
        const float y0 = o[nd][2 * half] * il, y1 = o[nd][2 * half + 1] * il;
        const uint32_t hv = pack2(y0, y1);
        *reinterpret_cast<uint32_t*>(a.out + base + d) = hv;
        if (a.out_lo) {
          const __half2 h2 = *reinterpret_cast<const __half2*>(&hv);
          const float2 hf = __half22float2(h2);
          *reinterpret_cast<uint32_t*>(a.out_lo + base + d) = pack2(y0 - hf.x, y1 - hf.y);
        }
      }
    }
    return;
  }

  // the cluster's partial states -> each CTA's own shared memory
  constexpr int RLD = S::RED_LD;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? rhi : rlo;
#pragma unroll
    for (int nd = 0; nd < ND; ++nd)
      *reinterpret_cast<float2*>(sRed + r * RLD + nd * 8 + tq * 2) = make_float2(o[nd][2 * half], o[nd][2 * half + 1]);
    if (tq == 0) sML[r] = half ? make_float2(m_hi, l_hi) : make_float2(m_lo, l_lo);
  }
  cluster_sync_all();
  // rank r combines rows [r * per, (r + 1) * per) of the tile
  const int per = (64 + csk - 1) / csk;
  const int rb = rank * per, re = min(rows, rb + per);
  constexpr int C4 = DH / 4;
  for (int idx = tid; idx < (re - rb) * C4; idx += 128) {
    const int r = rb + idx / C4, d = (idx % C4) * 4;
    float M = -INFINITY;
    for (int pr = 0; pr < csk; ++pr) {
      const float2 ml = dsmem_ld_f2(dsmem_addr(sML + r, pr));
      if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int pr = 0; pr < csk; ++pr) {
      const float2 ml = dsmem_ld_f2(dsmem_addr(sML + r, pr));
      if (!(ml.y > 0.f)) continue;
      const float w = exp2f(ml.x - M);
      const float4 v = dsmem_ld_f4(dsmem_addr(sRed + r * RLD + d, pr));
      L += w * ml.y;
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    const float il = L > 0.f ? 1.f / L : 0.f;
    const float y0 = acc.x * il, y1 = acc.y * il, y2 = acc.z * il, y3 = acc.w * il;
    const size_t base = static_cast<size_t>(qrow0 + r / G) * a.ld_out + (hk * G + r % G) * DH + d;
    const uint2 hv = make_uint2(pack2(y0, y1), pack2(y2, y3));
    *reinterpret_cast<uint2*>(a.out + base) = hv;
    if (a.out_lo) {
      const float2 h01 = __half22float2(*reinterpret_cast<const __half2*>(&hv.x));
      const float2 h23 = __half22float2(*reinterpret_cast<const __half2*>(&hv.y));
      *reinterpret_cast<uint2*>(a.out_lo + base) =
          make_uint2(pack2(y0 - h01.x, y1 - h01.y), pack2(y2 - h23.x, y3 - h23.y));
    }
  }
  cluster_sync_all();  // peers read this CTA's shared memory until here
}

template <int DH>
static int launch_tree_t(const TreeAttnArgs& a, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t r = cudaFuncSetAttribute(tree_attn_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TreeSmem<DH>::BYTES);
    if (r != cudaSuccess) return r;
    attr = true;
  }
  const dim3 grid(static_cast<unsigned>((a.n_br_tiles + a.n_pf_tiles) * a.csk), static_cast<unsigned>(a.Hkv), 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = TreeSmem<DH>::BYTES;
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
  return cudaLaunchKernelEx(&cfg, tree_attn_kernel<DH>, a);
}

int launch_tree_attention(const TreeAttnArgs& a, cudaStream_t s) {
  if (a.n_br_tiles + a.n_pf_tiles <= 0) return 0;
  if (a.csk < 1 || a.csk > 8) return cudaErrorInvalidValue;
  if (a.tpt < 1 || a.tpt * (a.Hq / a.Hkv) > 64) return cudaErrorInvalidValue;
  switch (a.DH) {
    case 16: return launch_tree_t<16>(a, s);
    case 64: return launch_tree_t<64>(a, s);
    case 128: return launch_tree_t<128>(a, s);
  }
  return cudaErrorInvalidValue;
}

int tree_attention_csk(int tiles, int Hkv, int max_blocks, int sms, bool tc) {
  static const int forced = [] {
    const char* e = std::getenv("PCD_TREE_CSK");
    return e ? std::atoi(e) : 0;
  }();
  if (forced >= 1 && forced <= 8) return forced;
  // Time model in microseconds: a CTA costs a fixed part, its share of the
  // tile's key blocks and, in a cluster, the combine; CTAs past what the SMs
  // hold at once run in a later wave.
  // fitted on GB300: the tensor-core kernel's start and epilogue ~6.6 us
  // (per-phase timer trace), ~2.4 us per 64-key block with the remainder MMAs
  // and gathered ancestor chunks, the cluster combine ~11 us (branch-pass
  // launches at key splits 1-4); the warp-MMA kernel's figures from
  // whole-launch times
  const double fixed = tc ? 6.6 : 3.0, per_block = tc ? 2.4 : 1.5, combine = tc ? 11.0 : 6.0;
  int best = 1;
  double best_t = 1e30;
  for (int csk = 1; csk <= 8 && csk <= max_blocks; ++csk) {
    const long long ctas = static_cast<long long>(tiles) * Hkv * csk;
    // resident CTAs: the tensor-core kernel runs one per SM, its clusters within a GPC each
    long long slots = static_cast<long long>(tc ? 1 : 2) * sms;
    if (tc) {
      const int q = tree_attention_tc_slots(csk);
      if (q > 0) slots = q;
    }
    const long long waves = (ctas + slots - 1) / slots;
    const int blocks = (max_blocks + csk - 1) / csk;
    const double t = static_cast<double>(waves) * (fixed + blocks * per_block + (csk > 1 ? combine : 0.0));
    if (t < best_t - 1e-9) {
      best_t = t;
      best = csk;
    }
  }
  return best;
}

}  // namespace pcd
