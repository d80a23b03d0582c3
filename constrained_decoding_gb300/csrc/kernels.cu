// Non-GEMM device steps of the PCD hot path: embedding gather, RMSNorm,
// RoPE + KV write, prefill / prefix attention, branch-ancestor merge,
// vocabulary log-sum-exp combine and field scoring.
#include <cfloat>
#include <cstdint>

#include "common.cuh"
#include "kernels.h"
#include "pcd.h"
#include "warp_mma.cuh"

namespace pcd {

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("PCD_PDL");
    return !e || std::atoi(e) != 0;
  }();
  return on;
}

// ======================================================================= embed
__global__ void embed_kernel(const int32_t* __restrict__ ids, int n, const act_t* __restrict__ E, int d, int vocab,
                             float* __restrict__ x, int* err) {
  griddep_launch_dependents();
  griddep_wait();
  const int t = blockIdx.x;
  if (t >= n) return;
  int id = ids[t];
  if (id < 0 || id >= vocab) {
    if (threadIdx.x == 0) record_error(err, DEV_BAD_INDEX);
    id = 0;
  }
  const uint4* src = reinterpret_cast<const uint4*>(E + static_cast<size_t>(id) * d);
  float4* dst = reinterpret_cast<float4*>(x + static_cast<size_t>(t) * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) {
    uint4 w = src[i];
    const __half2* h = reinterpret_cast<const __half2*>(&w);
    float2 a = __half22float2(h[0]), b = __half22float2(h[1]), c = __half22float2(h[2]),
           e = __half22float2(h[3]);
    dst[2 * i] = make_float4(a.x, a.y, b.x, b.y);
    dst[2 * i + 1] = make_float4(c.x, c.y, e.x, e.y);
  }
}

int launch_embed(const int32_t* ids, int n, const act_t* E, int d, int vocab, float* x, int* err, cudaStream_t s) {
  if (n <= 0) return 0;
  return launch_k(embed_kernel, dim3(n), dim3(128), 0, s, ids, n, E, d, vocab, x, err);
}

// ===================================================================== rmsnorm
// One CTA per row; the row stays in registers between the sum of squares and
// the scaling (fp32 statistics).
constexpr int kNormThreads = 256;
constexpr int kNormMaxVec = 8;  // float4 per thread: d <= 8192

__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const float* __restrict__ x, int ldx,
                                                               const int32_t* __restrict__ rows, int n, int d,
                                                               const float* __restrict__ gain, float eps,
                                                               act_t* __restrict__ out, int ldo,
                                                               act_t* __restrict__ out_lo) {
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x;
  const int src = rows ? rows[r] : r;
  const float4* xr = reinterpret_cast<const float4*>(x + static_cast<size_t>(src) * ldx);
  const int nv = d / 4;
  float4 v[kNormMaxVec];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kNormMaxVec; ++j) {
    const int i = threadIdx.x + j * kNormThreads;
    if (i < nv) {
      v[j] = xr[i];
      ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  __shared__ float red[kNormThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
  const float inv = rsqrtf(tot / static_cast<float>(d) + eps);
  const float4* g4 = reinterpret_cast<const float4*>(gain);
  uint2* o2 = reinterpret_cast<uint2*>(out + static_cast<size_t>(r) * ldo);
  uint2* l2 = out_lo ? reinterpret_cast<uint2*>(out_lo + static_cast<size_t>(r) * ldo) : nullptr;
#pragma unroll
  for (int j = 0; j < kNormMaxVec; ++j) {
    const int i = threadIdx.x + j * kNormThreads;
    if (i < nv) {
      const float4 g = g4[i];
      const float y0 = v[j].x * inv * g.x, y1 = v[j].y * inv * g.y, y2 = v[j].z * inv * g.z, y3 = v[j].w * inv * g.w;
      uint2 w;
      w.x = pack2(y0, y1);
      w.y = pack2(y2, y3);
      o2[i] = w;
      if (l2) {  // the rounding remainder, so hi + lo carries the fp32 value
        const __half2* h = reinterpret_cast<const __half2*>(&w);
        const float2 a = __half22float2(h[0]), b = __half22float2(h[1]);
        uint2 lo;
        lo.x = pack2(y0 - a.x, y1 - a.y);
        lo.y = pack2(y2 - b.x, y3 - b.y);
        l2[i] = lo;
      }
    }
  }
}

int launch_rmsnorm(const float* x, int ldx, const int32_t* rows, int n, int d, const float* gain, float eps, act_t* out,
                   int ldo, cudaStream_t s, act_t* out_lo) {
  if (n <= 0) return 0;
  if (d % 4 || d > 4 * kNormThreads * kNormMaxVec) return -1;
  return launch_k(rmsnorm_kernel, dim3(n), dim3(kNormThreads), 0, s, x, ldx, rows, n, d, gain, eps, out, ldo, out_lo);
}

// ====================================================================== rope_kv
// Rotate-half pairing (i, i + DH/2), angle pos * theta^(-2i/DH) from a
// (cos, sin) table built in double precision; four pairs per thread.
__global__ void rope_kv_kernel(RopeArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  // a thread takes four consecutive rotation pairs (i0 .. i0+3, i0+h .. i0+h+3
  // with h = DH/2) of one (token, head): 16-byte loads of q/k/v and of the
  // (cos, sin) table, 8-byte stores.  32-bit index arithmetic (the launcher
  // checks that every index fits).
  const unsigned half = static_cast<unsigned>(a.DH / 2);
  const unsigned quads = half / 4;
  const unsigned heads = static_cast<unsigned>(a.Hq + 2 * a.Hkv);
  const unsigned idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= static_cast<unsigned>(a.n) * heads * quads) return;
  const unsigned th = idx / quads;
  const int i0 = static_cast<int>(idx - th * quads) * 4;
  const int t = static_cast<int>(th / heads);
  const int h = static_cast<int>(th - static_cast<unsigned>(t) * heads);
  int pos = a.base + (a.rel ? a.rel[t] : t);
  if (pos < 0 || pos >= a.max_pos) {
    record_error(a.err, DEV_BAD_INDEX);
    pos = 0;
  }
  float4* src = reinterpret_cast<float4*>(const_cast<float*>(a.qkv) + static_cast<size_t>(t) * a.ldqkv + h * a.DH + i0);
  float4* src2 = src + half / 4;
  const float4 x1 = *src, x2 = *src2;
  if (a.clear_qkv) {  // leave the accumulation buffer zeroed for the next split-K projection
    *src = make_float4(0.f, 0.f, 0.f, 0.f);
    *src2 = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float y1[4] = {x1.x, x1.y, x1.z, x1.w}, y2[4] = {x2.x, x2.y, x2.z, x2.w};
  act_t *dst, *lo;
  size_t o;
  if (h < a.Hq + a.Hkv) {
    const float4* cp = reinterpret_cast<const float4*>(a.cs + static_cast<size_t>(pos) * half + i0);
    const float4 c01 = cp[0], c23 = cp[1];
    const float cs_c[4] = {c01.x, c01.z, c23.x, c23.z}, cs_s[4] = {c01.y, c01.w, c23.y, c23.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float u = y1[k], w = y2[k];
      y1[k] = u * cs_c[k] - w * cs_s[k];
      y2[k] = w * cs_c[k] + u * cs_s[k];
    }
    if (h < a.Hq) {
      o = (static_cast<size_t>(t) * a.Hq + h) * a.DH;
      dst = a.q;
      lo = a.q_lo;
    } else {
      o = (static_cast<size_t>(h - a.Hq) * a.kv_head_stride + a.kv_row0 + t) * a.DH;
      dst = a.k_dst;
      lo = a.k_lo;
    }
  } else {
    o = (static_cast<size_t>(h - a.Hq - a.Hkv) * a.kv_head_stride + a.kv_row0 + t) * a.DH;
    dst = a.v_dst;
    lo = a.v_lo;
  }
  const uint2 hv1 = make_uint2(pack2(y1[0], y1[1]), pack2(y1[2], y1[3]));
  const uint2 hv2 = make_uint2(pack2(y2[0], y2[1]), pack2(y2[2], y2[3]));
  *reinterpret_cast<uint2*>(dst + o + i0) = hv1;
  *reinterpret_cast<uint2*>(dst + o + half + i0) = hv2;
  if (lo) {  // value - fp16(value), itself rounded to fp16
    const __half* e1 = reinterpret_cast<const __half*>(&hv1);
    const __half* e2 = reinterpret_cast<const __half*>(&hv2);
    *reinterpret_cast<uint2*>(lo + o + i0) =
        make_uint2(pack2(y1[0] - a2f(e1[0]), y1[1] - a2f(e1[1])), pack2(y1[2] - a2f(e1[2]), y1[3] - a2f(e1[3])));
    *reinterpret_cast<uint2*>(lo + o + half + i0) =
        make_uint2(pack2(y2[0] - a2f(e2[0]), y2[1] - a2f(e2[1])), pack2(y2[2] - a2f(e2[2]), y2[3] - a2f(e2[3])));
  }
}

int launch_rope_kv(const RopeArgs& a, cudaStream_t s) {
  if (a.n <= 0) return 0;
  if (a.DH % 8 || a.ldqkv % 4) return cudaErrorInvalidValue;  // four pairs per thread, 16-byte rows
  const long long total = static_cast<long long>(a.n) * (a.Hq + 2 * a.Hkv) * (a.DH / 8);
  if (total >= (1ll << 31)) return cudaErrorInvalidValue;
  return launch_k(rope_kv_kernel, dim3(static_cast<unsigned>((total + 255) / 256)), dim3(256), 0, s, a);
}

// ==================================================================== attention
// Flash attention (online softmax, fp32 statistics) with mma.sync fp16
// tensor-core tiles.  A CTA owns 64 query rows of one KV head; the rows are
// (token, query head of the group) pairs, so every key tile loaded into
// shared memory serves all query heads that share it.  Key j is visible to a
// query at position p iff j <= p (causal prefill; branch queries sit after
// the whole prefix and see all of it).
template <int DH>
struct AttnSmem {
  static constexpr int LDS = DH + 8;  // padded row: conflict-free ldmatrix
  static constexpr int BYTES = (64 + 4 * 64) * LDS * 2 + 64 * 4;
};

template <int DH>
__global__ void __launch_bounds__(128) attn_kernel(AttnArgs a) {
  constexpr int LDS = AttnSmem<DH>::LDS;
  constexpr int KS = DH / 16;  // k-steps over the head dim
  constexpr int ND = DH / 8;   // 8-wide output column blocks
  extern __shared__ __align__(16) uint8_t attn_smem[];
  act_t* sQ = reinterpret_cast<act_t*>(attn_smem);
  act_t* sK = sQ + 64 * LDS;          // [2][64][LDS]
  act_t* sV = sK + 2 * 64 * LDS;      // [2][64][LDS]
  int* sPos = reinterpret_cast<int*>(sV + 2 * 64 * LDS);

  griddep_launch_dependents();
  griddep_wait();
  const int G = a.Hq / a.Hkv;
  const int rows = a.n_tok * G;
  const int nrb = gridDim.x;
  const int rb = a.causal_heavy_first ? (nrb - 1 - blockIdx.x) : blockIdx.x;
  const int hk = blockIdx.y;
  const int split = blockIdx.z;
  const int r0 = rb * 64;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tq = lane & 3;

  // query rows: positions, and the Q tile
  if (tid < 64) {
    const int r = r0 + tid;
    int p = -1;
    if (r < rows) {
      const int t = a.tok0 + r / G;
      p = a.base + (a.rel ? a.rel[t] : t);
    }
    sPos[tid] = p;
  }
  constexpr int QCH = DH / 8;  // 16-byte chunks per row
  for (int c = tid; c < 64 * QCH; c += 128) {
    const int rr = c / QCH, ch = c % QCH;
    const int r = r0 + rr;
    const bool ok = r < rows;
    const int t = a.tok0 + (ok ? r / G : 0), g = ok ? r % G : 0;
    const act_t* src = a.q + (static_cast<size_t>(t) * a.Hq + hk * G + g) * DH + ch * 8;
    cp_async16(sQ + rr * LDS + ch * 8, src, ok);
  }
  cp_async_commit();
  __syncthreads();
  int pmax = -1;
  for (int i = 0; i < 64; ++i) pmax = max(pmax, sPos[i]);
  const int k_lo = split * a.split_len;
  const int k_hi = min(min(a.n_keys, (split + 1) * a.split_len), pmax + 1);
  const int n_tiles = k_hi > k_lo ? (k_hi - k_lo + 63) / 64 : 0;

  const act_t* kbase = a.k + static_cast<size_t>(hk) * a.kv_head_stride * DH;
  const act_t* vbase = a.v + static_cast<size_t>(hk) * a.kv_head_stride * DH;
  auto load_kv = [&](int tile, int buf) {
    const int j0 = k_lo + tile * 64;
    for (int c = tid; c < 64 * QCH; c += 128) {
      const int kr = c / QCH, ch = c % QCH;
      const int j = j0 + kr;
      const bool ok = j < k_hi;
      const size_t off = static_cast<size_t>(ok ? j : 0) * DH + ch * 8;
      cp_async16(sK + (buf * 64 + kr) * LDS + ch * 8, kbase + off, ok);
      cp_async16(sV + (buf * 64 + kr) * LDS + ch * 8, vbase + off, ok);
    }
    cp_async_commit();
  };
  // Q fragments (the Q group was committed first)
  if (n_tiles > 0) {
    load_kv(0, 0);
    cp_async_wait<1>();
  } else {
    cp_async_wait<0>();
  }
  __syncthreads();
  uint32_t qf[KS][4];
#pragma unroll
  for (int kk = 0; kk < KS; ++kk)
    ldsm_x4(qf[kk], sQ + (warp * 16 + (lane & 15)) * LDS + kk * 16 + (lane >> 4) * 8);

  const int pos_lo = sPos[warp * 16 + gid], pos_hi = sPos[warp * 16 + gid + 8];
  float o[ND][4];
#pragma unroll
  for (int i = 0; i < ND; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

  for (int tile = 0; tile < n_tiles; ++tile) {
    const int buf = tile & 1;
    if (tile + 1 < n_tiles) {
      load_kv(tile + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const act_t* K = sK + buf * 64 * LDS;
    const act_t* V = sV + buf * 64 * LDS;
    const int j0 = k_lo + tile * 64;

    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int nb2 = 0; nb2 < 4; ++nb2) {
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        uint32_t b[4];
        ldsm_x4(b, K + (nb2 * 16 + (lane >> 4) * 8 + (lane & 7)) * LDS + kk * 16 + ((lane >> 3) & 1) * 8);
        mma16816(s[2 * nb2], qf[kk], b[0], b[1]);
        mma16816(s[2 * nb2 + 1], qf[kk], b[2], b[3]);
      }
    }
    // scale, mask, online softmax (log2 units)
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) {
      const int j = j0 + nb * 8 + tq * 2;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool in = (j + e) < k_hi;
        float v0 = s[nb][e] * a.scale_log2, v1 = s[nb][2 + e] * a.scale_log2;
        if (!in || j + e > pos_lo) v0 = -INFINITY;
        if (!in || j + e > pos_hi) v1 = -INFINITY;
        s[nb][e] = v0;
        s[nb][2 + e] = v1;
        mx_lo = fmaxf(mx_lo, v0);
        mx_hi = fmaxf(mx_hi, v1);
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
    for (int nb = 0; nb < 8; ++nb) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float p0 = (mn_lo == -INFINITY) ? 0.f : exp2f(s[nb][e] - mn_lo);
        const float p1 = (mn_hi == -INFINITY) ? 0.f : exp2f(s[nb][2 + e] - mn_hi);
        s[nb][e] = p0;
        s[nb][2 + e] = p1;
        rs_lo += p0;
        rs_hi += p1;
      }
    }
    l_lo = l_lo * c_lo + rs_lo;
    l_hi = l_hi * c_hi + rs_hi;
#pragma unroll
    for (int i = 0; i < ND; ++i) {
      o[i][0] *= c_lo;
      o[i][1] *= c_lo;
      o[i][2] *= c_hi;
      o[i][3] *= c_hi;
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
        uint32_t b[4];
        ldsm_x4_t(b, V + (kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7)) * LDS + nd2 * 16 + (lane >> 4) * 8);
        mma16816(o[2 * nd2], pa, b[0], b[1]);
        mma16816(o[2 * nd2 + 1], pa, b[2], b[3]);
      }
    }
    __syncthreads();  // the buffer is refilled next iteration
  }

  // finalise: full row sums across the quad
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, off);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, off);
  }
  const float il_lo = l_lo > 0.f ? 1.f / l_lo : 0.f;
  const float il_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
  const int rlo = r0 + warp * 16 + gid, rhi = rlo + 8;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? rhi : rlo;
    if (r >= rows) continue;
    const float il = half ? il_hi : il_lo;
    const int t = a.tok0 + r / G, g = r % G;
    if (!a.partial) {
      act_t* dst = a.out + static_cast<size_t>(t) * a.ld_out + (hk * G + g) * DH;
#pragma unroll
      for (int nd = 0; nd < ND; ++nd) {
        const int d = nd * 8 + tq * 2;
        *reinterpret_cast<uint32_t*>(dst + d) = pack2(o[nd][2 * half] * il, o[nd][2 * half + 1] * il);
      }
    } else {
      const size_t prow = (static_cast<size_t>(split) * a.Hkv + hk) * a.part_rows + static_cast<size_t>(t) * G + g;
      float* dst = a.part_o + prow * DH;
#pragma unroll
      for (int nd = 0; nd < ND; ++nd) {
        const int d = nd * 8 + tq * 2;
        *reinterpret_cast<float2*>(dst + d) = make_float2(o[nd][2 * half] * il, o[nd][2 * half + 1] * il);
      }
      if (tq == 0) a.part_ml[prow] = make_float2(half ? m_hi : m_lo, half ? l_hi : l_lo);
    }
  }
}

template <int DH>
static int launch_attn_t(const AttnArgs& a, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t r = cudaFuncSetAttribute(attn_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         AttnSmem<DH>::BYTES);
    if (r != cudaSuccess) return r;
    attr = true;
  }
  const int G = a.Hq / a.Hkv;
  const int rows = a.n_tok * G;
  dim3 grid((rows + 63) / 64, a.Hkv, a.n_splits);
  return launch_k(attn_kernel<DH>, grid, dim3(128), AttnSmem<DH>::BYTES, s, a);
}

int launch_attention(const AttnArgs& a, cudaStream_t s) {
  if (a.n_tok <= 0) return 0;
  switch (a.DH) {
    case 16: return launch_attn_t<16>(a, s);
    case 64: return launch_attn_t<64>(a, s);
    case 128: return launch_attn_t<128>(a, s);
  }
  return -1;
}

// ================================================================ branch merge
// One warp per (branch token, query head): merges the prefix partials of all
// key splits with the token's own ancestors in the branch (scaffold chain and
// trie path, the token itself included).  The ancestors' scores are computed
// by the lanes in parallel (lane j scores ancestor j), then each lane
// accumulates its DH/32 output dimensions over the weighted values.  With no
// ancestor list (anc_off == nullptr) it only combines the key splits.
template <int DH>
__global__ void __launch_bounds__(256) branch_merge_kernel(MergeArgs a) {
  constexpr int EPT = DH >= 32 ? DH / 32 : 1;
  __shared__ __align__(16) float sq[8][DH];
  griddep_launch_dependents();
  griddep_wait();
  const int wl = threadIdx.x >> 5;
  const int w = blockIdx.x * (blockDim.x >> 5) + wl;
  const int lane = threadIdx.x & 31;
  if (w >= a.n_tok * a.Hq) return;
  const int t = w / a.Hq, h = w % a.Hq;
  const int G = a.Hq / a.Hkv;
  const int hk = h / G, g = h % G;
  const int rows = a.n_tok * G;
  const int r = t * G + g;
  const act_t* qp = a.q + (static_cast<size_t>(t) * a.Hq + h) * DH;
  for (int d = lane; d < DH; d += 32) sq[wl][d] = a2f(qp[d]);
  __syncwarp();

  // prefix partials
  float m = -INFINITY, l = 0.f, acc[EPT];
#pragma unroll
  for (int i = 0; i < EPT; ++i) acc[i] = 0.f;
  for (int sp = 0; sp < a.n_splits; ++sp) {
    const size_t prow = (static_cast<size_t>(sp) * a.Hkv + hk) * rows + r;
    const float2 ml = a.part_ml[prow];
    if (!(ml.y > 0.f)) continue;
    const float mn = fmaxf(m, ml.x);
    const float co = exp2f(m - mn), cs = exp2f(ml.x - mn);
    const float* po = a.part_o + prow * DH;
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
      const int d = lane + 32 * i;
      acc[i] = acc[i] * co + (d < DH ? po[d] : 0.f) * ml.y * cs;
    }
    l = l * co + ml.y * cs;
    m = mn;
  }
  if (a.anc_off) {
    const int a0 = a.anc_off[t], a1 = a.anc_off[t + 1];
    for (int base = a0; base < a1; base += 32) {
      const int na = min(32, a1 - base);
      // lane j: score of ancestor base + j
      float sc = -INFINITY;
      int j = 0;
      if (lane < na) {
        j = a.anc_idx[base + lane];
        const uint4* kp = reinterpret_cast<const uint4*>(a.kb + (static_cast<size_t>(hk) * a.n_tok + j) * DH);
        float dot = 0.f;
#pragma unroll
        for (int c = 0; c < DH / 8; ++c) {
          const uint4 kv = kp[c];
          const __half2* k2 = reinterpret_cast<const __half2*>(&kv);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 kf = __half22float2(k2[e]);
            dot += sq[wl][c * 8 + 2 * e] * kf.x + sq[wl][c * 8 + 2 * e + 1] * kf.y;
          }
        }
        sc = dot * a.scale_log2;
      }
      float cm = sc;
#pragma unroll
      for (int o = 16; o; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
      const float mn = fmaxf(m, cm);
      const float co = exp2f(m - mn);
      const float p = lane < na ? exp2f(sc - mn) : 0.f;
      float ps = p;
#pragma unroll
      for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
#pragma unroll
      for (int i = 0; i < EPT; ++i) acc[i] *= co;
      l = l * co + ps;
      m = mn;
      for (int jj = 0; jj < na; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
        const int aj = __shfl_sync(0xffffffffu, j, jj);
        const act_t* vp = a.vb + (static_cast<size_t>(hk) * a.n_tok + aj) * DH;
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
          const int d = lane + 32 * i;
          if (d < DH) acc[i] += pj * a2f(vp[d]);
        }
      }
    }
  }
  const float il = l > 0.f ? 1.f / l : 0.f;
  act_t* dst = a.out + static_cast<size_t>(t) * a.ld_out + h * DH;
  act_t* dlo = a.out_lo ? a.out_lo + static_cast<size_t>(t) * a.ld_out + h * DH : nullptr;
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int d = lane + 32 * i;
    if (d < DH) {
      const float y = acc[i] * il;
      const act_t hv = f2a(y);
      dst[d] = hv;
      if (dlo) dlo[d] = f2a(y - a2f(hv));
    }
  }
}

int launch_branch_merge(const MergeArgs& a, cudaStream_t s) {
  const int warps = a.n_tok * a.Hq;
  if (warps <= 0) return 0;
  const int blocks = (warps + 7) / 8;
  switch (a.DH) {
    case 16: return launch_k(branch_merge_kernel<16>, dim3(blocks), dim3(256), 0, s, a);
    case 64: return launch_k(branch_merge_kernel<64>, dim3(blocks), dim3(256), 0, s, a);
    case 128: return launch_k(branch_merge_kernel<128>, dim3(blocks), dim3(256), 0, s, a);
  }
  return -1;
}

// ================================================================ lse combine
__global__ void lse_combine_kernel(const float2* __restrict__ part, int n_tiles, int R, float* __restrict__ lse) {
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= R) return;
  float m = -INFINITY;
  for (int i = lane; i < n_tiles; i += 32) m = fmaxf(m, part[static_cast<size_t>(i) * R + r].x);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float sum = 0.f;
  for (int i = lane; i < n_tiles; i += 32) {
    const float2 p = part[static_cast<size_t>(i) * R + r];
    sum += p.y * __expf(p.x - m);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) lse[r] = m + __logf(sum);
}

int launch_lse_combine(const float2* part, int n_tiles, int R, float* lse, cudaStream_t s) {
  if (R <= 0) return 0;
  return launch_k(lse_combine_kernel, dim3((R + 7) / 8), dim3(256), 0, s, part, n_tiles, R, lse);
}

// ====================================================================== score
// One CTA per field.  The full-vocabulary log-probability of a candidate path
// is ss_p = sum over the path of (z - lse).  The field's rule makes the path's
// score: sp_p = ss_p (sum), ss_p / path length (length-normalised mean), or
// the sum over the path of (z - log-sum-exp of the logits of the tokens
// allowed at that trie node) (per-level product of renormalised decisions).
// A label's score s_c is the log-sum-exp of the scores of the paths that
// spell it (one path per label unless the field lists spellings).  Then the
// candidate-only softmax of s at temperature T, the argmax (lowest index on
// ties), the top-2 margin of s, the candidate mass sum_p exp(ss_p) and the
// first-decision mass (distinct first tokens at the root readout row).
__global__ void __launch_bounds__(256) score_kernel(ScoreArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  const int f = blockIdx.x;
  const int c0 = a.fld_lab[f], c1 = a.fld_lab[f + 1];
  const int nl = c1 - c0;                                 // candidate paths
  const int o0 = a.fld_out[f], no = a.fld_out[f + 1] - o0;  // labels
  const float T = a.temp[f];
  const int rule = a.scoring[f];
  __shared__ float s_path[256];
  __shared__ int s_lab[256];
  __shared__ float red[32];
  __shared__ int redi[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;

  // path scores (more than 255 paths per field are rejected by the host)
  float sp = -INFINITY, ss = -INFINITY;
  if (tid < nl) {
    const int c = c0 + tid;
    const int i0 = a.lab_off[c], i1 = a.lab_off[c + 1];
    float acc = 0.f, lvl = 0.f;
    for (int i = i0; i < i1; ++i) {
      const int e = a.path[i];
      const int r = a.child_row[e];
      const float ze = a.z[e];
      acc += ze - a.lse[r];
      if (rule == PCD_SCORE_LEVEL) {
        // the node's allowed next tokens are its readout row's child entries
        const int e0 = a.row_ch[r], e1 = a.row_ch[r + 1];
        float m = -INFINITY;
        for (int x = e0; x < e1; ++x) m = fmaxf(m, a.z[x]);
        float sum = 0.f;
        for (int x = e0; x < e1; ++x) sum += __expf(a.z[x] - m);
        lvl += ze - (m + __logf(sum));
      }
    }
    ss = acc;
    sp = rule == PCD_SCORE_MEAN ? acc / static_cast<float>(i1 - i0) : (rule == PCD_SCORE_LEVEL ? lvl : acc);
    s_path[tid] = sp;
    s_lab[tid] = a.cand_label[c];
  }
  __syncthreads();
  // label scores: log-sum-exp over the label's spellings (exactly the path's
  // score when it has one)
  float sc = -INFINITY;
  if (tid < no) {
    float m = -INFINITY;
    for (int q = 0; q < nl; ++q)
      if (s_lab[q] == tid) m = fmaxf(m, s_path[q]);
    float sum = 0.f;
    for (int q = 0; q < nl; ++q)
      if (s_lab[q] == tid) sum += __expf(s_path[q] - m);
    sc = m + __logf(sum);
  }
  // block max of s (and its first index), block max of s/T
  auto block_max_idx = [&](float v, int idx, float& out_v, int& out_i) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
      if (ov > v || (ov == v && oi < idx)) v = ov, idx = oi;
    }
    if (lane == 0) red[warp] = v, redi[warp] = idx;
    __syncthreads();
    if (warp == 0) {
      v = lane < nw ? red[lane] : -INFINITY;
      idx = lane < nw ? redi[lane] : 0x7fffffff;
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
        if (ov > v || (ov == v && oi < idx)) v = ov, idx = oi;
      }
      if (lane == 0) red[0] = v, redi[0] = idx;
    }
    __syncthreads();
    out_v = red[0];
    out_i = redi[0];
    __syncthreads();
  };
  auto block_sum = [&](float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
      v = lane < nw ? red[lane] : 0.f;
#pragma unroll
      for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) red[0] = v;
    }
    __syncthreads();
    const float r = red[0];
    __syncthreads();
    return r;
  };
  float smax;
  int top;
  block_max_idx(sc, tid < no ? tid : 0x7fffffff, smax, top);
  // second best score: max over everything but the argmax
  float s2;
  int i2;
  block_max_idx((tid < no && tid != top) ? sc : -INFINITY, tid, s2, i2);
  // candidate mass from the full-vocabulary log-probs
  float ssmax;
  int ssi;
  block_max_idx(ss, tid, ssmax, ssi);
  const float es = tid < nl ? __expf(ss - ssmax) : 0.f;
  const float sum_es = block_sum(es);
  const float ea = tid < no ? __expf((sc - smax) / T) : 0.f;
  const float sum_ea = block_sum(ea);
  // first-decision mass at the field's root readout row
  const int root = a.fld_root[f];
  float fm = 0.f;
  for (int e = a.row_ch[root] + tid; e < a.row_ch[root + 1]; e += blockDim.x) fm += __expf(a.z[e] - a.lse[root]);
  fm = block_sum(fm);

  if (tid < no) {
    a.out_probs[o0 + tid] = ea / sum_ea;
    a.out_logprobs[o0 + tid] = sc;
  }
  if (tid == 0) {
    const float lm = ssmax + __logf(sum_es);
    float* o = a.out_field + static_cast<size_t>(f) * 8;
    o[0] = static_cast<float>(top);
    o[1] = __expf(lm);
    o[2] = lm;
    o[3] = no > 1 ? smax - s2 : INFINITY;
    o[4] = fm;
    o[5] = static_cast<float>(no);
    o[6] = 0.f;
    o[7] = 0.f;
  }
}

int launch_score(const ScoreArgs& a, cudaStream_t s) {
  if (a.n_fields <= 0) return 0;
  return launch_k(score_kernel, dim3(a.n_fields), dim3(256), 0, s, a);
}

}  // namespace pcd
