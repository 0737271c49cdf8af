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

#include <mutex>

#include "common.cuh"

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
};

template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  static CP_DEV void unpack(const uint4& u, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(h[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
};
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
// writes the final output and LSE and returns the counter to zero for the next call.  Publication follows the
// fence-then-count pattern: each CTA fences its partial before the atomic increment, and the
// last one fences again before reading the others' partials through L2.  No CTA waits on
// another, so nothing can stall.
template <typename T, int D, int G>
CP_DEV void fused_tail(const DecodeParams& p, int b, int g) {
  __shared__ int s_last;
  __shared__ float s_w[kMaxFusedPartials * G];  // per (partial, head): log2 LSE, then weight
  __shared__ float s_M[G], s_L[G];
  __syncthreads();
  const int P = p.cp * p.S;
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(p.counters + (long long)b * p.Hkv + g, 1);
    s_last = (prev == P - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const long long stride = (long long)p.B * p.Hq;           // between partials
  const long long unit0 = (long long)b * p.Hq + (long long)g * G;
  for (int i = threadIdx.x; i < P * G; i += blockDim.x)
    s_w[i] = __ldcg(p.lse + (i / G) * stride + unit0 + i % G) * kLog2e;
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
    if (threadIdx.x < G) p.lse[obase + threadIdx.x] = -INFINITY;
    if constexpr (FUSED) fused_tail<T, D, G>(p, b, g);
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
  if constexpr (FUSED) fused_tail<T, D, G>(p, b, g);

}

template <typename T, int D, bool F>
cudaError_t launch_g(const DecodeParams& p, int G, dim3 grid, cudaStream_t s) {
  switch (G) {
    case 1: decode_kernel<T, D, 1, F><<<grid, kWarps * 32, 0, s>>>(p); break;
    case 2: decode_kernel<T, D, 2, F><<<grid, kWarps * 32, 0, s>>>(p); break;
    case 4: decode_kernel<T, D, 4, F><<<grid, kWarps * 32, 0, s>>>(p); break;
    case 8: decode_kernel<T, D, 8, F><<<grid, kWarps * 32, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <bool F>
cudaError_t launch_all(const DecodeParams& p, const cp_decode_args& a, dim3 grid, cudaStream_t s) {
  const int G = a.num_q_heads / a.num_kv_heads;
  if (a.dtype == CP_BF16)
    return a.head_dim == 64 ? launch_g<__nv_bfloat16, 64, F>(p, G, grid, s)
                            : launch_g<__nv_bfloat16, 128, F>(p, G, grid, s);
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

// ------------------------------------------------------------------------------ no allocation
// Scratch for cp_decode_attention_noalloc: one array per GPU that loads this library, held until
// the process exits.  Host code must not use the symbol's host-side name as a device pointer;
// the device address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[CP_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's scratch array (the device must be current).
cudaError_t static_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = addr;
  }
  *ptr = g_scratch_addr[dev];
  return cudaSuccess;
}
}  // namespace

extern "C" cp_status cp_decode_attention_noalloc(const cp_decode_args* a, void* out,
                                                 float* out_lse, void* stream) {
  const cp_status st = cp_check_decode_args_for_fused(a, out);
  if (st != CP_OK) return st;
  size_t ol = 0, oo = 0;
  const size_t need = cp_decode_ws_layout(a->num_seqs, a->num_q_heads, a->num_kv_heads,
                                          a->head_dim, a->cp * a->num_splits, &ol, &oo);
  if (need > CP_NOALLOC_SCRATCH_BYTES)
    return cp_fail_detail(CP_ERR_INVALID_ARG,
                          "cp_decode_attention_noalloc needs %zu bytes of scratch but its static "
                          "array holds %zu: use fewer splits or a smaller batch",
                          need, (size_t)CP_NOALLOC_SCRATCH_BYTES);
  void* ws = nullptr;
  cudaError_t e = static_scratch(&ws);
  if (e != cudaSuccess) return cp_launch_status(e, "static scratch address");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the arrival counters must start at zero whatever an earlier call left behind
  e = cudaMemsetAsync(ws, 0, ol, s);
  if (e != cudaSuccess) return cp_launch_status(e, "static scratch clear");
  CpDecodeWorkspace w;
  w.counters = static_cast<int32_t*>(ws);
  w.partial_lse = reinterpret_cast<float*>(static_cast<char*>(ws) + ol);
  w.partial_out = reinterpret_cast<float*>(static_cast<char*>(ws) + oo);
  const float scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.f / sqrtf((float)a->head_dim);
  return cp_launch_status(cp_launch_decode_fused(*a, scale, w, out, out_lse, s),
                          "fused decode (static scratch) launch");
}
