// Decode partial attention over a round-robin paged kv cache ("allgather decode").
//
// "Add utility functions to enable pass-kv prefill and allgather decode" (vLLM PR 26059),
// Purpose: decode KV stays on the CP ranks round-robin, each rank attends the new query over
// its own tokens and the partials are combined (cp_lse_merge).  "[Feature] Prefill Context
// Parallel (PCP) basic support" (PR 28718), Purpose: per-rank block tables.
//
// Work unit (one CTA of 4 warps): split s of rank r's local tokens of sequence b, kv head g,
// all G query heads of that group.  The kernel is HBM-bound: every kv byte is read once with
// 16-byte loads straight into registers, a page (16 tokens, head-major so one head's page is
// contiguous) per warp per iteration, and all of a page's loads are issued before its math.
#include <math.h>

#include <cuda.h>

#include "common.cuh"
#include "sm100.cuh"

namespace cpattn {
namespace {

constexpr int kWarps = 4;
constexpr int kPage = 16;  // tokens per page (block_size)
constexpr int kMaxFusedPartials = 256;  // cp * splits of one fused decode call

struct DecodeParams {
  int B, Hq, Hkv, cp, I, S, ST, max_blocks;
  long long pool;
  float scale_log2;
  const void* q;
  const void* kc;
  const void* vc;
  const int32_t* tables;
  const int32_t* seq_lens;
  float* out;   // partials [cp*S][B][Hq][D] (the workspace when fused)
  float* lse;   // partial LSEs [cp*S][B][Hq]
  int32_t* err;
  // fused merge: per-(sequence, kv head) arrival counters, final output and LSE
  int32_t* counters;
  void* final_out;
  float* final_lse;
  // d = 128 tensor-core path: 1 = the maps are whole-page 3D boxes (one copy per page of K and
  // one of V), 0 = 2D boxes of 64 columns (two copies each)
  int page_box;
};

template <typename T> struct Vec;  // the CUDA-core kernel's 16-byte vector of T (f32 path)
template <> struct Vec<float> {
  static constexpr int N = 4;
  static CP_DEV void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
};

CP_DEV uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Fused merge (decode): after a CTA has written its partial it counts itself in for its
// (sequence, kv head); the CTA that arrives last merges the cp * splits partials of the G heads
// (the LSE merge: weights 2^(lse_p - M) staged once in shared memory, empty partials weigh 0),
// writes the final output and LSE and returns the counter to zero for the next call.
// Publication: after a CTA barrier (every thread's partial writes ordered before it), one thread
// counts the CTA in with an acquire-release atomic at GPU scope: its release side publishes the
// CTA's partial (cumulatively, through the barrier) and its acquire side lets the last CTA see
// every earlier CTA's partial; a second barrier passes that on to the last CTA's threads, which
// then read the partials through L2.  No CTA waits on another, so nothing can stall.
// Only the (rank, split) CTAs that hold tokens of the sequence (split * ST < the rank's share)
// count in and write a partial: an empty split returns at once, and the merge gives the
// partials it did not write weight 0.
CP_DEV bool split_live(const DecodeParams& p, int L, int part) {
  return (part % p.S) * (long long)p.ST < rank_local_len(L, part / p.S, p.cp, p.I);
}
CP_DEV int live_partials(const DecodeParams& p, int L) {
  int c = 0;
  for (int r = 0; r < p.cp; ++r) c += min(p.S, (rank_local_len(L, r, p.cp, p.I) + p.ST - 1) / p.ST);
  return c;
}
// s_w: shared scratch of kMaxFusedPartials * G floats, per (partial, head): log2 LSE, then
// weight.  The tensor-core kernel passes its K/V ring, idle by then, so that the merge adds no
// shared memory to the CTA (three CTAs per SM still fit at G = 16).
template <typename T, int D, int G>
CP_DEV void fused_tail(const DecodeParams& p, int b, int g, int L, float* s_w) {
  __shared__ int s_last;
  __shared__ float s_M[G], s_L[G];
  __syncthreads();
  const int P = p.cp * p.S;
  if (threadIdx.x == 0) {
    int prev;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(p.counters + (long long)b * p.Hkv + g)
                 : "memory");
    s_last = (prev == live_partials(p, L) - 1);
  }
  __syncthreads();
  if (!s_last) return;
  const long long stride = (long long)p.B * p.Hq;           // between partials
  const long long unit0 = (long long)b * p.Hq + (long long)g * G;
  for (int i = threadIdx.x; i < P * G; i += blockDim.x)
    s_w[i] = split_live(p, L, i / G) ? __ldcg(p.lse + (i / G) * stride + unit0 + i % G) * kLog2e
                                     : -INFINITY;
  __syncthreads();
  if (threadIdx.x < G) {
    float M = -INFINITY;
    for (int q = 0; q < P; ++q) M = fmaxf(M, s_w[q * G + threadIdx.x]);
    s_M[threadIdx.x] = M;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < P * G; i += blockDim.x) {
    const float M = s_M[i % G], lq = s_w[i];
    s_w[i] = (M > -INFINITY && lq > -INFINITY) ? exp2f(lq - M) : 0.f;
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float L = 0.f;
    for (int q = 0; q < P; ++q) L += s_w[q * G + threadIdx.x];
    s_L[threadIdx.x] = L;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int hh = i / D, dd = i % D;
    const float* src = p.out + (unit0 + hh) * D + dd;
    const long long pstride = stride * D;
    float acc = 0.f;
    int q = 0;
    for (; q + 8 <= P; q += 8) {  // eight partial rows in flight (empty ones weigh 0)
      float x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = __ldcg(src + (q + u) * pstride);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float w = s_w[(q + u) * G + hh];
        acc += w > 0.f ? w * x[u] : 0.f;
      }
    }
    for (; q < P; ++q) {
      const float w = s_w[q * G + hh];
      const float x = __ldcg(src + q * pstride);
      acc += w > 0.f ? w * x : 0.f;
    }
    const float L = s_L[hh];
    const float o = L > 0.f ? acc / L : 0.f;
    if constexpr (sizeof(T) == 2)
      static_cast<__nv_bfloat16*>(p.final_out)[(unit0 + hh) * D + dd] = __float2bfloat16_rn(o);
    else
      static_cast<float*>(p.final_out)[(unit0 + hh) * D + dd] = o;
    if (dd == 0 && p.final_lse)
      p.final_lse[unit0 + hh] = L > 0.f ? (s_M[hh] + log2f(L)) * kLn2 : -INFINITY;
  }
  if (threadIdx.x == 0) p.counters[(long long)b * p.Hkv + g] = 0;
}

// Fused decode, a CTA with no token of its sequence: it writes nothing and does not count in.
// Only a sequence without any token (seq_lens <= 0, outside the contract) has its first CTA
// write the exact result of no keys: zero output, LSE -inf.
template <typename T, int D, int G>
CP_DEV void fused_empty(const DecodeParams& p, int b, int g, int r, int split) {
  if (r != 0 || split != 0) return;
  const long long unit0 = (long long)b * p.Hq + (long long)g * G;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    if constexpr (sizeof(T) == 2)
      static_cast<__nv_bfloat16*>(p.final_out)[unit0 * D + i] = __float2bfloat16_rn(0.f);
    else
      static_cast<float*>(p.final_out)[unit0 * D + i] = 0.f;
  }
  if (threadIdx.x < G && p.final_lse) p.final_lse[unit0 + threadIdx.x] = -INFINITY;
}

template <typename T, int D, int G, bool FUSED>
__global__ void __launch_bounds__(kWarps * 32, 4) decode_kernel(const DecodeParams p) {
  constexpr int EPV = Vec<T>::N;          // elements per 16-byte vector
  constexpr int QKV = (D / 2) / EPV;      // K vectors per lane: token lane/2, vectors 2i+lane%2
  constexpr int NCH = D / EPV;            // V chunks per token
  constexpr int TG = 32 / NCH;            // token groups in a warp for P.V
  constexpr int TPL = kPage / TG;         // V tokens per lane
  static_assert(NCH <= 32 && 32 % NCH == 0, "head_dim / vector width");

  __shared__ __align__(16) float q_s[G][D];             // scaled into the log2 domain
  __shared__ __align__(16) float p_s[kWarps][kPage][G];
  __shared__ float m_w[kWarps][G], l_w[kWarps][G];
  __shared__ __align__(16) float o_w[kWarps][G][D];
  __shared__ float fused_w[FUSED ? kMaxFusedPartials * G : 1];  // the fused merge's weights

  const int split = blockIdx.x, g = blockIdx.y;
  // the cp ranks of a sequence are adjacent in launch order, so a (sequence, kv head) group's
  // CTAs run together and its fused merge is not deferred to the end of the grid
  const int r = blockIdx.z % p.cp, b = blockIdx.z / p.cp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = __ldg(p.seq_lens + b);
  const int n = rank_local_len(L, r, p.cp, p.I);
  const int l0 = split * p.ST;
  const int l1 = min(n, l0 + p.ST);
  const int part = r * p.S + split;
  const long long obase = ((long long)part * p.B + b) * p.Hq + (long long)g * G;

  if (l0 >= l1) {  // nothing of this rank falls in this split
    if constexpr (FUSED) fused_empty<T, D, G>(p, b, g, r, split);
    else if (threadIdx.x < G) p.lse[obase + threadIdx.x] = -INFINITY;
    return;
  }

  const T* qg = static_cast<const T*>(p.q) + ((long long)b * p.Hq + (long long)g * G) * D;
  for (int i = threadIdx.x; i < G * D; i += blockDim.x)
    (&q_s[0][0])[i] = Elem<T>::to_f(qg[i]) * p.scale_log2;
  __syncthreads();

  float m[G], l[G], acc[G][EPV];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    m[hh] = -INFINITY;
    l[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc[hh][e] = 0.f;
  }

  const int qk_tok = lane >> 1, half = lane & 1;
  const int v_ch = lane % NCH, v_tg = lane / NCH;
  const int32_t* trow = p.tables + ((long long)r * p.B + b) * p.max_blocks;
  const long long head_stride = (long long)kPage * D;  // elements of one head's page
  const T* kbase = static_cast<const T*>(p.kc);
  const T* vbase = static_cast<const T*>(p.vc);

  // This warp's pages: pg0 + warp, pg0 + warp + 4, ...  Their ids are fetched 32 at a time
  // (lane j holds the j-th), so no page waits on its table entry.
  const int pg0 = l0 / kPage, pg1 = (l1 + kPage - 1) / kPage;
  const int nmine = pg1 - pg0 > warp ? (pg1 - pg0 - warp + kWarps - 1) / kWarps : 0;

  auto page_id = [&](int j) -> int {  // j-th page of this warp (all lanes)
    const int pg = pg0 + warp + j * kWarps;
    int id = pg < p.max_blocks ? __ldg(trow + pg) : -1;
    if (id >= p.pool) id = -1;
    return id;
  };
  auto issue = [&](int id, uint4 (&kv)[QKV], uint4 (&vv)[TPL]) {
    if (id < 0) return;
    const long long off = (((long long)r * p.pool + id) * p.Hkv + g) * head_stride;
    const T* kp = kbase + off;
    const T* vp = vbase + off;
#pragma unroll
    for (int i = 0; i < QKV; ++i)
      kv[i] = ldg_stream(kp + (long long)qk_tok * D + (2 * i + half) * EPV);
#pragma unroll
    for (int i = 0; i < TPL; ++i)
      vv[i] = ldg_stream(vp + (long long)(v_tg + i * TG) * D + v_ch * EPV);
  };
  auto consume = [&](int j, int id, const uint4 (&kv)[QKV], const uint4 (&vv)[TPL]) {
    if (id < 0) {  // a table entry outside the pool: the page is skipped and reported
      if (lane == 0) report(p.err, CP_ERR_DEVICE_BOUNDS);
      return;
    }
    const int pg = pg0 + warp + j * kWarps;
    // scores of token qk_tok for the G heads (two lanes per token, one half of d each)
    float s[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) s[hh] = 0.f;
#pragma unroll
    for (int i = 0; i < QKV; ++i) {
      float kf[EPV];
      Vec<T>::unpack(kv[i], kf);
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float4* qv = reinterpret_cast<const float4*>(&q_s[hh][(2 * i + half) * EPV]);
#pragma unroll
        for (int e4 = 0; e4 < EPV / 4; ++e4) {
          const float4 qq = qv[e4];
          s[hh] += qq.x * kf[4 * e4] + qq.y * kf[4 * e4 + 1] + qq.z * kf[4 * e4 + 2] +
                   qq.w * kf[4 * e4 + 3];
        }
      }
    }
    const bool valid = pg * kPage + qk_tok < l1;
    float corr[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      s[hh] += __shfl_xor_sync(0xffffffffu, s[hh], 1);
      s[hh] = valid ? s[hh] : -INFINITY;
      const float m_new = fmaxf(m[hh], warp_max(s[hh]));
      corr[hh] = exp2f(m[hh] - m_new);
      const float pv = exp2f(s[hh] - m_new);
      l[hh] = l[hh] * corr[hh] + warp_sum(half == 0 ? pv : 0.f);
      m[hh] = m_new;
      if (half == 0) p_s[warp][qk_tok][hh] = pv;
    }
    __syncwarp();
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
      for (int e = 0; e < EPV; ++e) acc[hh][e] *= corr[hh];
#pragma unroll
    for (int i = 0; i < TPL; ++i) {
      float vf[EPV];
      Vec<T>::unpack(vv[i], vf);
      const int t = v_tg + i * TG;
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float pw = p_s[warp][t][hh];
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[hh][e] += pw * vf[e];
      }
    }
    __syncwarp();
  };

  for (int j0 = 0; j0 < nmine; j0 += 32) {
    const int cnt = min(32, nmine - j0);
    const int my_id = lane < cnt ? page_id(j0 + lane) : -1;
    for (int j = 0; j < cnt; ++j) {
      const int id = __shfl_sync(0xffffffffu, my_id, j);
      uint4 kv[QKV], vv[TPL];
      issue(id, kv, vv);
      consume(j0 + j, id, kv, vv);
    }
  }

  // token groups of the warp -> one partial per warp
#pragma unroll
  for (int hh = 0; hh < G; ++hh)
#pragma unroll
    for (int e = 0; e < EPV; ++e)
#pragma unroll
      for (int o = NCH; o < 32; o <<= 1) acc[hh][e] += __shfl_xor_sync(0xffffffffu, acc[hh][e], o);
  if (lane == 0) {
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      m_w[warp][hh] = m[hh];
      l_w[warp][hh] = l[hh];
    }
  }
  if (v_tg == 0) {
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
      for (int e = 0; e < EPV; ++e) o_w[warp][hh][v_ch * EPV + e] = acc[hh][e];
  }
  __syncthreads();

  // warps -> the CTA's partial (warps that saw no page carry m = -inf and weight 0)
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int hh = i / D, dd = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, m_w[w][hh]);
    float Ls = 0.f, Os = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float e = exp2f(m_w[w][hh] - M);
      Ls += e * l_w[w][hh];
      Os += e * o_w[w][hh][dd];
    }
    if (Ls > 0.f) {
      p.out[(obase + hh) * D + dd] = Os / Ls;
      if (dd == 0) p.lse[obase + hh] = (M + log2f(Ls)) * kLn2;
    } else if (dd == 0) {
      p.lse[obase + hh] = -INFINITY;
    }
  }
  if constexpr (FUSED) fused_tail<T, D, G>(p, b, g, L, fused_w);

}

// ------------------------------------------------------------------------------ tensor-core decode
// bf16 decode with the kv bytes moved by TMA and the arithmetic on tensor cores.  Per CTA:
// 4 consumer warps and 1 producer warp, three CTAs per SM.  The producer streams every page's K
// and V rows of one kv head (16 tokens x d, one whole-page box each, or two 2D boxes of 64
// columns; 128-byte swizzle) into a 2-stage ring per consumer warp.  A consumer computes, for
// its page,
//   S = Q K^T   with mma.sync m16n8k16: A = the G query heads (rows >= G are zero) kept in
//               registers for the whole CTA, B = K from shared memory via ldmatrix;
//   P           online softmax per head, in the fragment the MMA left it in (a row = a head,
//               so the 16 tokens of a head live in the 4 lanes of a quad: two shuffles);
//   O += P V    A = P (that same fragment, rounded to bf16), B = V via ldmatrix.trans.
// The swizzled layout makes every ldmatrix phase touch 8 distinct bank groups.
// Three CTAs of 2-stage rings per SM keep as many bytes in flight as two of 3-stage rings, and
// one CTA's end (its partial's writes, the fused form's release and merge) then idles a third
// of the SM's streams instead of half: measured 6.60 -> 6.68 TB/s (partials), 6.35 -> 6.64
// (fused) on the 64-sequence decode.  It caps a thread at 128 registers (a few spilled words).
constexpr int kCW = 4;  // consumer warps
constexpr int kST = 2;  // ring stages per consumer warp
constexpr long long kDecodeBudget = 4000000000ll;  // SM cycles per wait (~2 s)

template <int D>
struct MLayout {
  static constexpr int kPageBytes = kPage * D * 2;  // one head's K (or V) rows of a page
  static constexpr int kStage = 2 * kPageBytes;
  static constexpr int oRing = 0;
  static constexpr int kRing = kCW * kST * kStage;
  static constexpr int oM = kRing;                  // m [kCW][16] (one per MMA row)
  static constexpr int oL = oM + kCW * 16 * 4;      // l [kCW][16]
  static constexpr int oBar = oL + kCW * 16 * 4;
  static constexpr int nBar = 2 * kCW * kST;        // full, empty
  static constexpr int oFlag = oBar + nBar * 8;     // page valid [kCW][kST], abort
  static constexpr int kBytes = oFlag + (kCW * kST + 1) * 4;
  static constexpr int kAlloc = kBytes + 1024;      // base rounded up to the 1 KB swizzle atom
  static_assert(kCW * 16 * D * 4 <= kRing, "warp partials reuse the ring");
  static_assert(kMaxFusedPartials * 16 * 4 <= kRing, "the fused merge's weights reuse the ring");
  static_assert(kAlloc + 1024 <= 232448, "shared memory per CTA");
};

CP_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
CP_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
// D (16x8 f32) += A (16x16 bf16, rows gid / gid+8) * B (16x8 bf16).  a1, a3 (rows 8-15) are 0
// when at most 8 query heads share the kv head.
CP_DEV void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                     uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Byte address of the 16-byte chunk holding (token t, dim d) in a 128B-swizzled page half-box.
CP_DEV uint32_t page_addr(uint32_t base, int t, int d) {
  return base + (uint32_t)((d >> 6) * (kPage * 128) + t * 128 + ((((d & 63) >> 3) ^ (t & 7)) << 4));
}

template <int D, int G, bool FUSED>
__global__ void __launch_bounds__((kCW + 1) * 32, 3)
    decode_mma_kernel(const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v, const DecodeParams p) {
  using T = __nv_bfloat16;
  using Ly = MLayout<D>;
  constexpr int KB = D / 64;  // 64-column boxes per page row
  static_assert(G <= 16, "query heads per kv head (MMA rows)");
  constexpr bool TWO = G > 8;  // rows gid + 8 hold heads 8 .. G-1
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = sm100::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sb = smem_raw + (base - raw);
  float* m_w = reinterpret_cast<float*>(sb + Ly::oM);
  float* l_w = reinterpret_cast<float*>(sb + Ly::oL);
  volatile int* flags = reinterpret_cast<volatile int*>(sb + Ly::oFlag);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sb + Ly::oFlag + kCW * kST * 4);
  auto full = [&](int w, int s) -> uint32_t { return base + Ly::oBar + 8u * (uint32_t)(w * kST + s); };
  auto empty = [&](int w, int s) -> uint32_t {
    return base + Ly::oBar + 8u * (uint32_t)(kCW * kST + w * kST + s);
  };
  auto slot = [&](int w, int s) -> uint32_t { return base + Ly::oRing + (uint32_t)((w * kST + s) * Ly::kStage); };

  const int split = blockIdx.x, g = blockIdx.y;
  const int r = blockIdx.z % p.cp, b = blockIdx.z / p.cp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = __ldg(p.seq_lens + b);
  const int n = rank_local_len(L, r, p.cp, p.I);
  const int l0 = split * p.ST;
  const int l1 = min(n, l0 + p.ST);
  const int part = r * p.S + split;
  const long long obase = ((long long)part * p.B + b) * p.Hq + (long long)g * G;
  if (l0 >= l1) {  // nothing of this rank falls in this split
    if constexpr (FUSED) fused_empty<T, D, G>(p, b, g, r, split);
    else if (threadIdx.x < G) p.lse[obase + threadIdx.x] = -INFINITY;
    return;
  }
  if (threadIdx.x == 0) {
    for (int w = 0; w < kCW; ++w)
      for (int s = 0; s < kST; ++s) {
        sm100::mbar_init(full(w, s), 1);
        sm100::mbar_init(empty(w, s), 1);
      }
    *abort_flag = 0u;
    sm100::fence_mbar_init();
  }
  __syncthreads();

  const int pg0 = l0 / kPage, pg1 = (l1 + kPage - 1) / kPage;
  const int npages = pg1 - pg0;
  const int32_t* trow = p.tables + ((long long)r * p.B + b) * p.max_blocks;

  if (warp == kCW) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      sm100::tma_prefetch_desc(&map_k);
      sm100::tma_prefetch_desc(&map_v);
    }
    int issued = 0;
    bool ok = true;
    for (int j0 = 0; ok && j0 < npages; j0 += 32) {
      const int cnt = min(32, npages - j0);
      int my_id = -1;
      if (lane < cnt) {
        const int pg = pg0 + j0 + lane;
        my_id = pg < p.max_blocks ? __ldg(trow + pg) : -1;
        if (my_id >= p.pool || my_id < 0) my_id = -1;
      }
      for (int i = 0; i < cnt; ++i) {
        const int id = __shfl_sync(0xffffffffu, my_id, i);
        int good = 1;
        if (lane == 0) {
          const int j = j0 + i, w = j % kCW, k = j / kCW, st = k % kST;
          const uint32_t ph = (uint32_t)(k / kST) & 1u;
          if (!sm100::mbar_wait(empty(w, st), ph ^ 1u, abort_flag, kDecodeBudget)) {
            good = 0;
          } else {
            flags[w * kST + st] = id >= 0;
            if (id >= 0) {
              const int y = (int)((((long long)r * p.pool + id) * p.Hkv + g) * kPage);
              const uint32_t ks = slot(w, st);
              sm100::mbar_expect_tx(full(w, st), 2 * Ly::kPageBytes);
              if (KB == 2 && p.page_box) {  // [half][16 rows][128 B], the layout read below
                sm100::tma_load_3d(ks, &map_k, 0, y, 0, full(w, st));
                sm100::tma_load_3d(ks + Ly::kPageBytes, &map_v, 0, y, 0, full(w, st));
              } else {
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
                  sm100::tma_load_2d(ks + kb * (kPage * 128), &map_k, kb * 64, y, full(w, st));
                  sm100::tma_load_2d(ks + Ly::kPageBytes + kb * (kPage * 128), &map_v, kb * 64, y,
                                     full(w, st));
                }
              }
            } else {  // a table entry outside the pool: the page is skipped and reported
              report(p.err, CP_ERR_DEVICE_BOUNDS);
              sm100::mbar_arrive(full(w, st));  // the consumer sees flag 0 and skips the page
            }
            issued = j + 1;
          }
        }
        if (!__shfl_sync(0xffffffffu, good, 0)) {
          ok = false;
          break;
        }
      }
    }
    if (lane == 0) {
      if (!ok) {
        *abort_flag = 1u;
        report(p.err, CP_ERR_TIMEOUT);
      }
      // drain: every copy issued into this CTA's shared memory has landed before it exits
      for (int j = max(0, issued - kCW * kST); j < issued; ++j) {
        const int w = j % kCW, k = j / kCW;
        sm100::mbar_wait(full(w, k % kST), (uint32_t)(k / kST) & 1u, nullptr, kDecodeBudget);
      }
    }
  }

  const int gid = lane >> 2, tid = lane & 3;  // MMA fragment row (head) and column pair
  float o[D / 8][4];
  float m = -INFINITY, l = 0.f, m2 = -INFINITY, l2 = 0.f;  // rows gid and gid + 8
#pragma unroll
  for (int nb = 0; nb < D / 8; ++nb)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nb][e] = 0.f;
  if (warp < kCW) {
    // ------------------------------------------------------------------ consumers
    // Q rows as MMA A fragments (bf16 pairs straight from memory; rows >= G are zero)
    uint32_t qa0[D / 16], qa2[D / 16], qa1[D / 16], qa3[D / 16];
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        static_cast<const T*>(p.q) + ((long long)b * p.Hq + (long long)g * G + gid) * D);
    const uint32_t* qrow8 = qrow + 8 * (D / 2);  // head gid + 8
#pragma unroll
    for (int ds = 0; ds < D / 16; ++ds) {
      qa0[ds] = gid < G ? __ldg(qrow + ds * 8 + tid) : 0u;
      qa2[ds] = gid < G ? __ldg(qrow + ds * 8 + 4 + tid) : 0u;
      qa1[ds] = TWO && gid + 8 < G ? __ldg(qrow8 + ds * 8 + tid) : 0u;
      qa3[ds] = TWO && gid + 8 < G ? __ldg(qrow8 + ds * 8 + 4 + tid) : 0u;
    }
    const float sc = p.scale_log2;
    const int li = lane >> 3, lj = lane & 7;  // ldmatrix: matrix and row this lane addresses
    const int nmine = npages > warp ? (npages - warp + kCW - 1) / kCW : 0;
    for (int k = 0; k < nmine; ++k) {
      const int st = k % kST;
      const bool ok = __all_sync(0xffffffffu, sm100::mbar_wait(full(warp, st), (uint32_t)(k / kST) & 1u,
                                                               abort_flag, kDecodeBudget));
      if (!ok) {
        if (lane == 0) {
          *abort_flag = 1u;
          report(p.err, CP_ERR_TIMEOUT);
        }
        break;
      }
      const int pg = pg0 + warp + k * kCW;
      if (flags[warp * kST + st]) {
        const uint32_t kp = slot(warp, st), vp = kp + Ly::kPageBytes;
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};  // tokens 0-7, 8-15
#pragma unroll
        for (int ds = 0; ds < D / 16; ++ds) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(page_addr(kp, ((li >> 1) << 3) + lj, ds * 16 + ((li & 1) << 3)), b0, b1, b2, b3);
          mma16816(s0, qa0[ds], qa1[ds], qa2[ds], qa3[ds], b0, b1);
          mma16816(s1, qa0[ds], qa1[ds], qa2[ds], qa3[ds], b2, b3);
        }
        // head gid, tokens 2tid, 2tid+1, 8+2tid, 9+2tid of this page
        const int t0 = pg * kPage + 2 * tid;
        float x0 = t0 < l1 ? s0[0] * sc : -INFINITY;
        float x1 = t0 + 1 < l1 ? s0[1] * sc : -INFINITY;
        float x2 = t0 + 8 < l1 ? s1[0] * sc : -INFINITY;
        float x3 = t0 + 9 < l1 ? s1[1] * sc : -INFINITY;
        float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m, mx);
        const float corr = m_new == -INFINITY ? 1.f : exp2f(m - m_new);
        const float p0 = x0 == -INFINITY ? 0.f : exp2f(x0 - m_new);
        const float p1 = x1 == -INFINITY ? 0.f : exp2f(x1 - m_new);
        const float p2 = x2 == -INFINITY ? 0.f : exp2f(x2 - m_new);
        const float p3 = x3 == -INFINITY ? 0.f : exp2f(x3 - m_new);
        float ps = (p0 + p1) + (p2 + p3);
        ps += __shfl_xor_sync(0xffffffffu, ps, 1);
        ps += __shfl_xor_sync(0xffffffffu, ps, 2);
        l = l * corr + ps;
        m = m_new;
        __nv_bfloat162 pa = __floats2bfloat162_rn(p0, p1), pb = __floats2bfloat162_rn(p2, p3);
        const uint32_t pa0 = *reinterpret_cast<uint32_t*>(&pa), pa2 = *reinterpret_cast<uint32_t*>(&pb);
        uint32_t pa1 = 0u, pa3 = 0u;
        float corr2 = 1.f;
        if constexpr (TWO) {  // the same online softmax for head gid + 8 (fragment elements 2, 3)
          const float y0 = t0 < l1 ? s0[2] * sc : -INFINITY;
          const float y1 = t0 + 1 < l1 ? s0[3] * sc : -INFINITY;
          const float y2 = t0 + 8 < l1 ? s1[2] * sc : -INFINITY;
          const float y3 = t0 + 9 < l1 ? s1[3] * sc : -INFINITY;
          float my = fmaxf(fmaxf(y0, y1), fmaxf(y2, y3));
          my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 1));
          my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 2));
          const float m2_new = fmaxf(m2, my);
          corr2 = m2_new == -INFINITY ? 1.f : exp2f(m2 - m2_new);
          const float q0 = y0 == -INFINITY ? 0.f : exp2f(y0 - m2_new);
          const float q1 = y1 == -INFINITY ? 0.f : exp2f(y1 - m2_new);
          const float q2 = y2 == -INFINITY ? 0.f : exp2f(y2 - m2_new);
          const float q3 = y3 == -INFINITY ? 0.f : exp2f(y3 - m2_new);
          float qs = (q0 + q1) + (q2 + q3);
          qs += __shfl_xor_sync(0xffffffffu, qs, 1);
          qs += __shfl_xor_sync(0xffffffffu, qs, 2);
          l2 = l2 * corr2 + qs;
          m2 = m2_new;
          __nv_bfloat162 qa = __floats2bfloat162_rn(q0, q1), qb = __floats2bfloat162_rn(q2, q3);
          pa1 = *reinterpret_cast<uint32_t*>(&qa);
          pa3 = *reinterpret_cast<uint32_t*>(&qb);
        }
#pragma unroll
        for (int nb = 0; nb < D / 8; ++nb) {
          o[nb][0] *= corr;
          o[nb][1] *= corr;
          if constexpr (TWO) {
            o[nb][2] *= corr2;
            o[nb][3] *= corr2;
          }
        }
#pragma unroll
        for (int nb = 0; nb < D / 16; ++nb) {
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(page_addr(vp, ((li & 1) << 3) + lj, nb * 16 + ((li >> 1) << 3)), v0, v1, v2, v3);
          mma16816(o[2 * nb], pa0, pa1, pa2, pa3, v0, v1);
          mma16816(o[2 * nb + 1], pa0, pa1, pa2, pa3, v2, v3);
        }
      } else if (lane == 0) {
        report(p.err, CP_ERR_DEVICE_BOUNDS);
      }
      __syncwarp();
      if (lane == 0) sm100::mbar_arrive(empty(warp, st));
    }
  }
  __syncthreads();  // all pages consumed and all copies landed: the ring is free

  // warps -> one partial for the CTA (o_w reuses the ring)
  float* o_w = reinterpret_cast<float*>(sb + Ly::oRing);
  if (warp < kCW && gid < G) {
    if (tid == 0) {
      m_w[warp * 16 + gid] = m;
      l_w[warp * 16 + gid] = l;
    }
#pragma unroll
    for (int nb = 0; nb < D / 8; ++nb) {
      o_w[(warp * G + gid) * D + nb * 8 + 2 * tid] = o[nb][0];
      o_w[(warp * G + gid) * D + nb * 8 + 2 * tid + 1] = o[nb][1];
    }
  }
  if constexpr (TWO) {
    if (warp < kCW && gid + 8 < G) {
      if (tid == 0) {
        m_w[warp * 16 + gid + 8] = m2;
        l_w[warp * 16 + gid + 8] = l2;
      }
#pragma unroll
      for (int nb = 0; nb < D / 8; ++nb) {
        o_w[(warp * G + gid + 8) * D + nb * 8 + 2 * tid] = o[nb][2];
        o_w[(warp * G + gid + 8) * D + nb * 8 + 2 * tid + 1] = o[nb][3];
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int hh = i / D, dd = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCW; ++w) M = fmaxf(M, m_w[w * 16 + hh]);
    float Ls = 0.f, Os = 0.f;
#pragma unroll
    for (int w = 0; w < kCW; ++w) {
      const float mw = m_w[w * 16 + hh];
      const float e = mw > -INFINITY ? exp2f(mw - M) : 0.f;
      Ls += e * l_w[w * 16 + hh];
      Os += e * o_w[(w * G + hh) * D + dd];
    }
    if (Ls > 0.f) {
      p.out[(obase + hh) * D + dd] = Os / Ls;
      if (dd == 0) p.lse[obase + hh] = (M + log2f(Ls)) * kLn2;
    } else if (dd == 0) {
      p.lse[obase + hh] = -INFINITY;
    }
  }
  // the merge weights go to the K/V ring: free once every warp has passed fused_tail's barrier
  // (the warp partials read above live there too)
  if constexpr (FUSED) fused_tail<T, D, G>(p, b, g, L, reinterpret_cast<float*>(sb + Ly::oRing));
}

template <int D, bool F>
cudaError_t launch_mma_g(const DecodeParams& p, int G, dim3 grid, const CUtensorMap& mk,
                         const CUtensorMap& mv, cudaStream_t s) {
  auto go = [&](auto kern) -> cudaError_t {
    const int smem = MLayout<D>::kAlloc;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, (kCW + 1) * 32, smem, s>>>(mk, mv, p);
    return cudaGetLastError();
  };
  switch (G) {  // query heads per kv head = MMA rows in use (of 8)
    case 1: return go(decode_mma_kernel<D, 1, F>);
    case 2: return go(decode_mma_kernel<D, 2, F>);
    case 3: return go(decode_mma_kernel<D, 3, F>);
    case 4: return go(decode_mma_kernel<D, 4, F>);
    case 5: return go(decode_mma_kernel<D, 5, F>);
    case 6: return go(decode_mma_kernel<D, 6, F>);
    case 7: return go(decode_mma_kernel<D, 7, F>);
    case 8: return go(decode_mma_kernel<D, 8, F>);
    case 9: return go(decode_mma_kernel<D, 9, F>);
    case 10: return go(decode_mma_kernel<D, 10, F>);
    case 11: return go(decode_mma_kernel<D, 11, F>);
    case 12: return go(decode_mma_kernel<D, 12, F>);
    case 13: return go(decode_mma_kernel<D, 13, F>);
    case 14: return go(decode_mma_kernel<D, 14, F>);
    case 15: return go(decode_mma_kernel<D, 15, F>);
    case 16: return go(decode_mma_kernel<D, 16, F>);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int D, bool F>
cudaError_t launch_g(const DecodeParams& p, int G, dim3 grid, cudaStream_t s) {
  switch (G) {
    case 1: decode_kernel<T, D, 1, F><<<grid, kWarps * 32, 0, s>>>(p); break;
    case 2: decode_kernel<T, D, 2, F><<<grid, kWarps * 32, 0, s>>>(p); break;
    case 3: decode_kernel<T, D, 3, F><<<grid, kWarps * 32, 0, s>>>(p); break;
    case 4: decode_kernel<T, D, 4, F><<<grid, kWarps * 32, 0, s>>>(p); break;
    case 5: decode_kernel<T, D, 5, F><<<grid, kWarps * 32, 0, s>>>(p); break;
    case 6: decode_kernel<T, D, 6, F><<<grid, kWarps * 32, 0, s>>>(p); break;
    case 7: decode_kernel<T, D, 7, F><<<grid, kWarps * 32, 0, s>>>(p); break;
    case 8: decode_kernel<T, D, 8, F><<<grid, kWarps * 32, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <bool F>
cudaError_t launch_all(const DecodeParams& p0, const cp_decode_args& a, dim3 grid, cudaStream_t s) {
  const int G = a.num_q_heads / a.num_kv_heads;
  DecodeParams p = p0;
  p.page_box = 0;
  if (a.dtype == CP_BF16) {  // tensor-core kernel with TMA-staged pages
    CUtensorMap mk, mv;
    const unsigned long long rows = (unsigned long long)a.cp * a.pool_pages * a.num_kv_heads * kPage;
    // d = 128: one whole-page box per page of K and of V (half the copies of 64-column boxes;
    // the copy engine's per-box cost bounds this kernel), else 64-column boxes
    if (a.head_dim == 128 && cp_make_bf16_page_map(&mk, a.k_cache, rows) &&
        cp_make_bf16_page_map(&mv, a.v_cache, rows)) {
      p.page_box = 1;
    } else if (!cp_make_bf16_map_2d(&mk, a.k_cache, a.head_dim, rows, a.head_dim, kPage) ||
               !cp_make_bf16_map_2d(&mv, a.v_cache, a.head_dim, rows, a.head_dim, kPage)) {
      return cudaErrorInvalidValue;
    }
    return a.head_dim == 64 ? launch_mma_g<64, F>(p, G, grid, mk, mv, s)
                            : launch_mma_g<128, F>(p, G, grid, mk, mv, s);
  }
  return a.head_dim == 64 ? launch_g<float, 64, F>(p, G, grid, s) : launch_g<float, 128, F>(p, G, grid, s);
}

DecodeParams make_params(const cp_decode_args& a, float scale) {
  DecodeParams p;
  p.B = a.num_seqs;
  p.Hq = a.num_q_heads;
  p.Hkv = a.num_kv_heads;
  p.cp = a.cp;
  p.I = a.interleave;
  p.S = a.num_splits;
  p.ST = a.split_tokens;
  p.max_blocks = a.max_blocks;
  p.pool = a.pool_pages;
  p.scale_log2 = scale * kLog2e;
  p.q = a.q;
  p.kc = a.k_cache;
  p.vc = a.v_cache;
  p.tables = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.out = a.out;
  p.lse = a.lse;
  p.err = a.err;
  p.counters = nullptr;
  p.final_out = nullptr;
  p.final_lse = nullptr;
  p.page_box = 0;
  return p;
}

}  // namespace
}  // namespace cpattn

cudaError_t cp_launch_decode(const cp_decode_args& a, float scale, cudaStream_t s) {
  using namespace cpattn;
  const DecodeParams p = make_params(a, scale);
  dim3 grid(a.num_splits, a.num_kv_heads, a.cp * a.num_seqs);
  return launch_all<false>(p, a, grid, s);
}

cudaError_t cp_launch_decode_fused(const cp_decode_args& a, float scale, const CpDecodeWorkspace& ws,
                                   void* out, float* out_lse, cudaStream_t s) {
  using namespace cpattn;
  DecodeParams p = make_params(a, scale);
  p.out = ws.partial_out;
  p.lse = ws.partial_lse;
  p.counters = ws.counters;
  p.final_out = out;
  p.final_lse = out_lse;
  dim3 grid(a.num_splits, a.num_kv_heads, a.cp * a.num_seqs);
  return launch_all<true>(p, a, grid, s);
}
