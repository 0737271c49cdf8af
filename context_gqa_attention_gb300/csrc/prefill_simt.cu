// Partial attention on CUDA cores: one warp per (query row, query head), lanes split the
// head dimension, keys streamed one at a time with an online softmax.
//
// This is the plain path: it serves f32 inputs and acts as an independent cross-check of
// the tensor-core kernel.  Pairs follow "Add utility functions to enable pass-kv prefill and
// allgather decode" (vLLM PR 26059), Purpose: pass-KV (kv shard s = chunks s, 2cp-1-s) and
// pass-Q (kv rank r = round-robin resident tokens).
#include "common.cuh"

namespace cpattn {
namespace {

struct SimtParams {
  int mode, B, Nq, Hq, Hkv, cp, I, bs, max_blocks, q_shard, kv_shard;
  long long pool;
  float scale_log2;
  const int32_t* cu_q;
  const int32_t* cu_kv;  // pass-KV: kv rows per sequence (null: the query rows)
  const int32_t* seq_lens_kv;
  const void* q;
  const void* k;
  const void* v;
  const int32_t* tables;
  float* out;
  float* lse;
  int32_t* err;
};

template <typename T, int D>
struct Acc {
  static constexpr int E = D / 32;
  float m = -INFINITY, l = 0.f, o[E];
  float q[E];
  CP_DEV void init() {
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = 0.f;
    m = -INFINITY;
    l = 0.f;
  }
  CP_DEV void key(const T* __restrict__ krow, const T* __restrict__ vrow, int lane) {
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) part += q[e] * Elem<T>::to_f(krow[lane * E + e]);
    const float s = warp_sum(part);               // log2-domain score
    const float m_new = fmaxf(m, s);
    const float corr = exp2f(m - m_new);          // 0 when m = -inf
    const float p = exp2f(s - m_new);
    l = l * corr + p;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = o[e] * corr + p * Elem<T>::to_f(vrow[lane * E + e]);
    m = m_new;
  }
};

template <typename T, int D>
__global__ void __launch_bounds__(256) prefill_simt_kernel(const SimtParams p) {
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= (long long)p.Nq * p.Hq) return;
  const int row = (int)(warp / p.Hq);
  const int h = (int)(warp % p.Hq);
  const int b = seq_of_row(p.cu_q, p.B, row);
  const int q0 = p.cu_q[b];
  const int Tq = p.cu_q[b + 1] - q0;
  const int t = row - q0;
  const int cp = p.cp;
  if (p.q_shard >= 0 && shard_of_chunk(chunk_of(t, Tq, cp), cp) != p.q_shard) return;
  const int g = h / (p.Hq / p.Hkv);
  constexpr int E = D / 32;

  Acc<T, D> acc;
  const T* qrow = static_cast<const T*>(p.q) + ((long long)row * p.Hq + h) * D;
#pragma unroll
  for (int e = 0; e < E; ++e) acc.q[e] = Elem<T>::to_f(qrow[lane * E + e]) * p.scale_log2;

  const int p_lo = p.kv_shard >= 0 ? p.kv_shard : 0;
  const int p_hi = p.kv_shard >= 0 ? p.kv_shard + 1 : cp;
  for (int part = p_lo; part < p_hi; ++part) {
    acc.init();
    bool bad = false;
    if (p.mode == CP_PASS_KV) {
      const T* K = static_cast<const T*>(p.k);
      const T* V = static_cast<const T*>(p.v);
      // kv tokens of the sequence (cached + new); this query sits at position C + t
      const int kv0 = p.cu_kv ? p.cu_kv[b] : q0;
      const int Tkv = p.cu_kv ? p.cu_kv[b + 1] - kv0 : Tq;
      const int C = Tkv - Tq;
      if (C < 0) bad = true;  // fewer kv tokens than new queries: flagged, the row skipped
      const int chunks[2] = {part, 2 * cp - 1 - part};
      for (int ci = 0; ci < 2 && !bad; ++ci) {
        const int c = chunks[ci];
        const int ks = chunk_bound(c, Tkv, cp);
        const int ke = min(chunk_bound(c + 1, Tkv, cp), C + t + 1);
        for (int j = ks; j < ke; ++j) {
          const long long kr = ((long long)(kv0 + j) * p.Hkv + g) * D;
          acc.key(K + kr, V + kr, lane);
        }
      }
    } else {
      const T* Kc = static_cast<const T*>(p.k);
      const T* Vc = static_cast<const T*>(p.v);
      const long long L = p.seq_lens_kv[b];
      if (L < Tq) bad = true;  // fewer kv tokens than new queries: flagged, the row skipped
      const long long qpos = L - Tq + t;
      const int n = rank_local_len(qpos + 1, part, cp, p.I);
      const int32_t* trow = p.tables + ((long long)part * p.B + b) * p.max_blocks;
      for (int l = 0; l < n; ++l) {
        const int col = l / p.bs;
        const int page = col < p.max_blocks ? __ldg(trow + col) : -1;
        if (page < 0 || page >= p.pool) { bad = true; break; }
        const long long kr = ((((long long)part * p.pool + page) * p.Hkv + g) * p.bs + (l % p.bs)) * D;
        acc.key(Kc + kr, Vc + kr, lane);
      }
    }
    if (bad) {
      if (lane == 0) report(p.err, CP_ERR_DEVICE_BOUNDS);
      continue;
    }
    const long long orow = ((long long)part * p.Nq + row) * p.Hq + h;
    if (acc.l > 0.f) {
      const float inv = 1.f / acc.l;
#pragma unroll
      for (int e = 0; e < E; ++e) p.out[orow * D + lane * E + e] = acc.o[e] * inv;
      if (lane == 0) p.lse[orow] = (acc.m + log2f(acc.l)) * kLn2;
    } else if (lane == 0) {
      p.lse[orow] = -INFINITY;
    }
  }
}

}  // namespace
}  // namespace cpattn

cudaError_t cp_launch_prefill_simt(const cp_prefill_args& a, float scale, cudaStream_t s) {
  using namespace cpattn;
  SimtParams p;
  p.mode = a.mode;
  p.B = a.num_seqs;
  p.Hq = a.num_q_heads;
  p.Hkv = a.num_kv_heads;
  p.cp = a.cp;
  p.I = a.interleave;
  p.bs = a.block_size;
  p.max_blocks = a.max_blocks;
  p.q_shard = a.q_shard;
  p.kv_shard = a.kv_shard;
  p.pool = a.pool_pages;
  p.scale_log2 = scale * kLog2e;
  p.cu_q = a.cu_seqlens_q;
  p.cu_kv = a.mode == CP_PASS_KV ? a.cu_seqlens_kv : nullptr;
  p.seq_lens_kv = a.seq_lens_kv;
  p.q = a.q;
  p.k = a.mode == CP_PASS_KV ? a.k : a.k_cache;
  p.v = a.mode == CP_PASS_KV ? a.v : a.v_cache;
  p.tables = a.block_tables;
  p.out = a.out;
  p.lse = a.lse;
  p.err = a.err;
  p.Nq = a.total_q;
  const long long warps = (long long)p.Nq * p.Hq;
  if (warps == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
  if (a.dtype == CP_F32) {
    if (a.head_dim == 64) prefill_simt_kernel<float, 64><<<blocks, 256, 0, s>>>(p);
    else prefill_simt_kernel<float, 128><<<blocks, 256, 0, s>>>(p);
  } else {
    if (a.head_dim == 64) prefill_simt_kernel<__nv_bfloat16, 64><<<blocks, 256, 0, s>>>(p);
    else prefill_simt_kernel<__nv_bfloat16, 128><<<blocks, 256, 0, s>>>(p);
  }
  return cudaGetLastError();
}
