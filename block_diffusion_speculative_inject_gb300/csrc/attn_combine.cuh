// The split-KV merge of one query row, shared by the combine kernel and the tensor-core
// split kernel's fused combine. A warp merges row r (query head g = r / Q of the kv head,
// block row j = r % Q) of request b: the context splits' (max m_s, sum l_s, unnormalised
// partial output acc_s) and the block's own K+1 keys and values (fp32 q/k/v rows, staged in
// shared memory by stage_block_kv), in log2 units:
//   o = (sum_s acc_s 2^(m_s - M) + sum_kk 2^(s_kk - M) v_kk) / (sum_s l_s 2^(m_s - M) + sum_kk 2^(s_kk - M))
// Each lane scores one block key and owns HD/32 output dimensions; every load of the row is
// issued before any is used, and the order of every sum is fixed.
#pragma once
#include "common.cuh"

namespace dflash {

template <int HD>
struct CombineSmem {
  static constexpr int KP = HD + 1;               // padded rows: lane-per-key reads are conflict free
  float *ks;                                      // [32][KP] block keys
  float *vs;                                      // [32][HD] block values
};

// Block K/V of (request b, kv head kvh) into shared memory: float4 loads, all issued first.
template <int HD>
__device__ __forceinline__ void stage_block_kv(int b, int kvh, int nq, int nkv, int Q, const float *qkv,
                                               CombineSmem<HD> sm, int tid, int nthreads) {
  constexpr int V4 = HD / 4, KP = CombineSmem<HD>::KP;
  const int qkv_dim = (nq + 2 * nkv) * HD;
  for (int i0 = 0; i0 < Q * V4; i0 += 4 * nthreads) {
    float4 kv4[4], vv4[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + tid + u * nthreads;       // float4 index over [Q][HD/4]
      const int kk = i / V4, d4 = i % V4;
      const bool in = kk < Q;
      const float4 *row = (const float4 *)(qkv + ((size_t)b * Q + (in ? kk : 0)) * qkv_dim + (size_t)nq * HD);
      kv4[u] = in ? row[(size_t)kvh * V4 + d4] : make_float4(0.f, 0.f, 0.f, 0.f);
      vv4[u] = in ? row[(size_t)(nkv + kvh) * V4 + d4] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + tid + u * nthreads;
      const int kk = i / V4, d4 = i % V4;
      if (kk < Q) {
        const float4 a = kv4[u], v = vv4[u];
        sm.ks[kk * KP + 4 * d4 + 0] = a.x; sm.ks[kk * KP + 4 * d4 + 1] = a.y;
        sm.ks[kk * KP + 4 * d4 + 2] = a.z; sm.ks[kk * KP + 4 * d4 + 3] = a.w;
        *(float4 *)&sm.vs[kk * HD + 4 * d4] = v;
      }
    }
  }
}

// The loads of one row, issued before any of them is used (so that the caller can stage the
// block K/V meanwhile). MS >= the request's split count; qs: the warp's HD floats of shared
// memory (the q row). With coherent = true the partials are read at L2 (they were written
// by other CTAs of the same grid).
template <int HD, int MS>
struct CombineRow {
  float ms, ls;
  float po[MS][HD / 32];
};

template <int HD, int MS, bool coherent>
__device__ __forceinline__ void combine_load(CombineRow<HD, MS> &cr, int r, int b, int kvh, int nq, int nkv, int Q,
                                             int ns, int max_split, const float *part_o, const float *part_ml,
                                             const float *qkv, float *qs, int lane) {
  constexpr int DPL = HD / 32;
  const int G = nq / nkv, qkv_dim = (nq + 2 * nkv) * HD;
  const int g = r / Q, j = r % Q, h = kvh * G + g;
  const size_t row = (size_t)b * Q + j;
  const size_t base = (row * nq + h) * max_split;
  auto ld = [&](const float *p) { return coherent ? __ldcg(p) : *p; };
#pragma unroll
  for (int d = 0; d < DPL; ++d) qs[lane + 32 * d] = qkv[row * qkv_dim + (size_t)h * HD + lane + 32 * d];
  cr.ms = -INFINITY;
  cr.ls = 0.f;
  if (lane < ns) {
    cr.ms = ld(part_ml + (base + lane) * 2);
    cr.ls = ld(part_ml + (base + lane) * 2 + 1);
  }
#pragma unroll
  for (int sp = 0; sp < MS; ++sp)
#pragma unroll
    for (int d = 0; d < DPL; ++d) cr.po[sp][d] = sp < ns ? ld(part_o + (base + sp) * HD + lane + 32 * d) : 0.f;
}

// The merge itself, once the block K/V (and this warp's q row) are in shared memory.
template <int HD, int MS>
__device__ __forceinline__ void combine_finish(const CombineRow<HD, MS> &cr, int r, int b, int kvh, int nq, int nkv,
                                               int Q, int ns, float scale_log2, int causal, OpOut o,
                                               CombineSmem<HD> sm, const float *qs, int lane) {
  constexpr int DPL = HD / 32, KP = CombineSmem<HD>::KP;
  const int G = nq / nkv;
  const int g = r / Q, j = r % Q, h = kvh * G + g;
  const size_t row = (size_t)b * Q + j;
  // block key `lane` is seen by this row unless the causal variant hides keys after it
  const bool see = lane < Q && (!causal || lane <= j);
  float sk = -INFINITY;
  if (see) {
    float t = 0.f;
#pragma unroll 16
    for (int d = 0; d < HD; ++d) t = fmaf(qs[d], sm.ks[lane * KP + d], t);
    sk = t * scale_log2;
  }
  const float M = warp_max(fmaxf(sk, cr.ms));
  const float pk = see ? exp2f(sk - M) : 0.f;
  const float cs = lane < ns ? exp2f(cr.ms - M) : 0.f;
  const float Lsum = warp_sum(pk + cs * cr.ls);
  float acc[DPL] = {};
#pragma unroll
  for (int sp = 0; sp < MS; ++sp) {
    const float c = __shfl_sync(0xffffffffu, cs, sp);     // 0 for sp >= ns
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[d] = fmaf(c, cr.po[sp][d], acc[d]);
  }
  for (int kk = 0; kk < Q; ++kk) {
    const float p = __shfl_sync(0xffffffffu, pk, kk);
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[d] = fmaf(p, sm.vs[kk * HD + lane + 32 * d], acc[d]);
  }
  const float inv = 1.f / Lsum;
  const size_t dst = row * (nq * HD) + (size_t)h * HD;
#pragma unroll
  for (int d = 0; d < DPL; ++d) write_op(o, dst + lane + 32 * d, acc[d] * inv);
}

}  // namespace dflash
