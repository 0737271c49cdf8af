// Partial attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), bf16 in,
// f32 accumulate.
//
// Pairs: "Add utility functions to enable pass-kv prefill and allgather decode" (vLLM PR
// 26059), Purpose -- pass-KV (Q tile of chunk c against kv shard s = chunks s, 2cp-1-s) and
// pass-Q (Q tile against kv rank r's round-robin resident tokens in paged storage, "[Feature]
// Prefill Context Parallel (PCP) basic support" (PR 28718), Purpose: per-rank block tables).
//
// Two kernels.  prefill_tc2_kernel (the default) runs two "tiles" per CTA -- two query heads of
// one kv group, or for odd G two consecutive 128-row tiles of one head -- against one kv shard
// / rank (or, fused, against all of them):
//   warp 0      TMA producer: both Q tiles once, then K and V tiles (128 keys) through a
//               4-slot ring; paged kv arrives one box per page.
//   warp 1      TMEM owner and MMA issuer (one thread): S = Q K^T into the tile's TMEM S
//               columns, then O += P V with P read from TMEM; order per key tile
//               PV0(t) | QK0(t+1) | PV1(t) | QK1(t+1), so each tile's softmax overlaps the
//               other tile's two MMAs.
//   warps 2-3   idle (they complete the first warpgroup, whose register budget is lowered so
//               that the softmax warpgroups can raise theirs)
//   warps 4-11  two softmax warpgroups, one per tile: thread i owns query row i (TMEM lane i),
//               reads its S row with tcgen05.ld, masks by position, keeps the running max /
//               sum, rescales O in TMEM only when the max grows by more than 2^8, writes P
//               (bf16) back over its S columns, and finally normalises O and writes the output
//               and its LSE (rows staged in shared memory, then one whole row per warp store).
// prefill_tc1_kernel (CP_IMPL_TCGEN05_SINGLE) runs one head per CTA with a 2-stage ring and P
// in shared memory.
// Every wait is bounded; on expiry the CTA raises CP_ERR_TIMEOUT, drains its own copies and
// MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "sm100.cuh"

namespace cpattn {
namespace {

using namespace sm100;

constexpr int BM = 128;          // query rows per tile (TMEM lanes)
constexpr int BN = 128;          // keys per tile
constexpr int NS = 2;            // K/V pipeline stages (the drain below assumes 2)
constexpr int kThreads = 192;
constexpr long long kBudget = 4000000000ll;  // SM cycles per wait (~2 s)
constexpr float kRescaleThreshold = 8.f;     // log2 units

// Division of a numerator below 2^31 by a divisor fixed for the launch as one multiply and one
// shift (Granlund and Montgomery, "Division by invariant integers using multiplication", 1994,
// with 31-bit numerators): l = ceil(log2 d), m = ceil(2^(31+l) / d) < 2^32, then
// n / d = (n m) >> (31 + l).  The work-item decode at a CTA's start runs a chain of such
// divisions before its first load can be addressed.
struct FastDiv {
  uint32_t d, m, s;
};
inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  const unsigned long long num = 1ull << (31 + l);
  return FastDiv{d, (uint32_t)((num + d - 1) / d), 31 + l};
}
CP_DEV uint32_t fdiv(uint32_t n, const FastDiv& f) {
  return (uint32_t)(((unsigned long long)n * f.m) >> f.s);
}
// n / f.d, by the multiply and shift (FAST) or by plain integer division: the fused pass-Q
// kernel keeps the plain division, measured faster there (with the constants its spills grew).
template <bool FAST>
CP_DEV uint32_t udiv(uint32_t n, const FastDiv& f) {
  if constexpr (FAST) return fdiv(n, f);
  else return n / f.d;
}

struct TcParams {
  int mode, B, Hq, Hkv, cp, I, max_blocks, q_shard, kv_shard, TPC, Nq, debug;
  // pass-KV partials: head groups outermost within a sequence (see decode_work_at)
  int heads_outer;
  // divisors of the work-item decode: item groups of heads, q slots (2 cp TPC), cp, TPC, 2 cp
  // (chunk bounds), G (q heads per kv head)
  FastDiv f_groups, f_nslot, f_cp, f_tpc, f_2cp, f_G;
  long long pool, budget;
  float scale_log2;
  const int32_t* cu_q;
  const int32_t* cu_kv;     // pass-KV: kv rows per sequence (null: the query rows)
  const int32_t* seq_lens_kv;
  const int32_t* tables;
  float* out;
  float* lse;
  int32_t* err;
  // fused pass-KV: one item covers every kv shard (keys [0, q_hi)) and writes the final bf16
  // output [Nq][Hq][d] and LSE [Nq][Hq] instead of partials
  int fused;
  __nv_bfloat16* out_final;
  float* lse_final;
  // 1: the output base is 16-byte aligned, so a warp's full group of 32 rows goes out through
  // its shared-memory staging buffer as whole-row stores
  int row_out;
  // fused pass-Q, split tail: CTAs past the first n_whole run one of split_k rank ranges of
  // item n_whole + (CTA - n_whole) / split_k and write its normalised rows and LSEs to
  // ws_out [piece][2][BM][d] / ws_lse [piece][2][BM] (piece = CTA - n_whole; 2 = the CTA's
  // tiles) for fq_split_merge_kernel.  split_k <= 1: every item runs whole.
  int n_whole, split_k;
  float* ws_out;
  float* ws_lse;
};

template <int D>
struct Layout {
  static constexpr int kQ = BM * D * 2;
  static constexpr int kKV = BN * D * 2;
  static constexpr int kP = BM * BN * 2;
  static constexpr int oQ = 0;
  static constexpr int oK = oQ + kQ;
  static constexpr int oV = oK + NS * kKV;
  static constexpr int oP = oV + NS * kKV;
  static constexpr int oBar = oP + kP;
  static constexpr int bQ = 0, bKF = 1, bVF = bKF + NS, bKE = bVF + NS, bVE = bKE + NS,
                       bS = bVE + NS, bP = bS + 2, bO = bP + 1, bDone = bO + 1, nBar = bDone + 1;
  static constexpr int oMisc = oBar + nBar * 8;
  static constexpr int kBytes = oMisc + 16;
  // +1 KB so the base can be rounded up to the 1 KB swizzle-atom alignment; never below
  // 120 KB so that a single CTA (and its 512 TMEM columns) occupies an SM.
  static constexpr int kAlloc = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
  static_assert(kAlloc <= 232448, "dynamic shared memory beyond the 227 KB per-CTA limit");
};

struct Work {
  int valid, b, h, g, p;
  int q_row0, q_lo, q_hi;   // first token-major row; tile rows [q_lo, q_hi) of the sequence
  long long qpos0;          // position of row q_lo (cached context + q_lo)
  int kv_row0;              // pass-KV: first token-major kv row of the sequence
  int ks[2], ke[2], nt[2];  // pass-KV key ranges (positions) and their tile counts
  int n_local;              // pass-Q: resident tokens of rank p that any row can see
  int r_lo, r_hi;           // fused pass-Q: the ranks the item walks
  int ntiles;
};

// pass-Q: block-table entries of key tile t (NP pages of 16 rank-local tokens).  Entries past
// the table's width read as -1; rows past the rank's visible tokens are not loaded.
template <int NP>
CP_DEV void fetch_page_ids(const int32_t* trow, int t, int n_local, int max_blocks, int (&id)[NP]) {
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    const int col = t * NP + j;
    id[j] = (col * 16 < n_local && col < max_blocks) ? __ldg(trow + col) : -1;
  }
}

// Tensor-map row of each page of key tile t.  A visible page whose entry is outside the pool
// flags CP_ERR_DEVICE_BOUNDS; it and the pages past the visible range reload the tile's last
// valid page (finite data, masked by the softmax) so every stage receives the same byte count.
template <int NP>
CP_DEV void page_rows(const int (&id)[NP], int t, int n_local, long long pool, int Hkv, int rank, int g,
                      int* err, int (&row)[NP]) {
  int last_good = -1;
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    int pg = -1;
    if ((t * NP + j) * 16 < n_local) {
      pg = id[j];
      if (pg < 0 || pg >= pool) {
        report(err, CP_ERR_DEVICE_BOUNDS);
        pg = -1;
      }
    }
    if (pg >= 0) last_good = pg;
    row[j] = pg;
  }
  if (last_good < 0) last_good = 0;
#pragma unroll
  for (int j = 0; j < NP; ++j)
    row[j] = (int)((((long long)rank * pool + (row[j] >= 0 ? row[j] : last_good)) * Hkv + g) * 16);
}

// Fused pass-Q: key tile t of an item -> (rank r, tile tr within r's resident tokens), walked in
// order (ranks with no visible token skipped).  n_r: r's resident tokens any row of the item
// sees (kv_end = position after the item's last query).
struct RankWalk {
  int r, tr, nt_r, n_r;
};
// Tokens of rank r among positions [0, L) of the round-robin deal (as rank_local_len) for the
// positions the kernel sees: L <= seq_lens_kv < 2^31, with g = min(I cp, 2^31), so one 32-bit
// division and no 64-bit fallback in the loops that walk ranks.
CP_DEV int rank_len32(long long L, int r, int I, uint32_t g) {
  const uint32_t l = (uint32_t)L, q = l / g, rem = l - q * g;
  const long long x = (long long)rem - (long long)r * I;
  return (int)(q * (uint32_t)I) + (int)(x < 0 ? 0 : (x > I ? I : x));
}

CP_DEV void walk_settle(RankWalk& k, long long kv_end, int cp, int I, int r_end) {
  const uint32_t g = (long long)I * cp < (1ll << 31) ? (uint32_t)(I * cp) : (1u << 31);
  while (k.tr >= k.nt_r && k.r + 1 < r_end) {
    ++k.r;
    k.n_r = rank_len32(kv_end, k.r, I, g);
    k.nt_r = (k.n_r + BN - 1) / BN;
    k.tr = 0;
  }
}
CP_DEV RankWalk walk_start(long long kv_end, int cp, int I, int r_lo, int r_end) {
  RankWalk k{r_lo - 1, 0, 0, 0};
  walk_settle(k, kv_end, cp, I, r_end);
  return k;
}
CP_DEV void walk_next(RankWalk& k, long long kv_end, int cp, int I, int r_end) {
  ++k.tr;
  walk_settle(k, kv_end, cp, I, r_end);
}

// Chunk bound floor(k T / 2cp) (as chunk_bound) with the launch's divisor constants.
template <bool FAST>
CP_DEV int chunk_bound_f(int k, int T, const TcParams& p) {
  if constexpr (FAST) {
    const unsigned long long num = (unsigned long long)k * (unsigned)T;
    if (num < 0x80000000ull) return (int)fdiv((uint32_t)num, p.f_2cp);
  }
  return chunk_bound(k, T, p.cp);
}

// Work item index -> (q tile slot, sequence, kv shard, head group of `hpc` consecutive q heads).
// Slots run heaviest first (last chunk, last tile) so long items start early.
// `span` query rows per item: BM (one tile; head pairs) or 2 BM (two tiles of one head).
// Fused pass-Q items walk ranks [r_lo, r_hi) (all of them unless the item is split).
template <bool FAST = true>
CP_DEV Work decode_work_at(const TcParams& p, unsigned lin, int hpc, int span = BM, int r_lo = 0,
                           int r_hi = 1 << 30) {
  Work w;
  w.valid = 0;
  w.r_lo = r_lo;
  w.r_hi = min(r_hi, p.cp);
  // the item space is below 2^31; p.f_groups divides by Hq / hpc
  const unsigned groups = (unsigned)(p.Hq / hpc);
  const unsigned nslot = 2u * (unsigned)p.cp * (unsigned)p.TPC;
  unsigned q;
  int slot;
  if (p.heads_outer) {
    // pass-KV partials with a sequence's K/V larger than L2 can hold beside the outgoing
    // partial rows: kv shard fastest, then slot (heaviest first), then head group, so the CTAs
    // resident at one time read one kv head's K/V of one sequence
    q = udiv<FAST>(lin, p.f_cp);
    w.p = (int)(lin - q * (unsigned)p.cp);
    lin = q;
    q = udiv<FAST>(lin, p.f_nslot);
    slot = (int)(lin - q * nslot);
    lin = q;
    q = udiv<FAST>(lin, p.f_groups);
    w.h = (int)(lin - q * groups) * hpc;
    w.b = (int)q;
  } else {
  q = udiv<FAST>(lin, p.f_groups);
  w.h = (int)(lin - q * groups) * hpc;
  lin = q;
  if (p.mode == CP_PASS_Q) {
    // pass-Q items cost about the same (every query sees its rank's whole cached context), so
    // they run sequence by sequence and rank by rank: the CTAs resident at one time read the
    // pages of one or two (sequence, rank) pairs, which stay in L2
    q = udiv<FAST>(lin, p.f_nslot);
    slot = (int)(lin - q * nslot);
    lin = q;
    if (p.kv_shard >= 0 || p.fused) {
      w.p = p.fused ? 0 : p.kv_shard;
    } else {
      q = udiv<FAST>(lin, p.f_cp);
      w.p = (int)(lin - q * (unsigned)p.cp);
      lin = q;
    }
    w.b = (int)lin;
  } else {
    // pass-KV: sequence by sequence, each heaviest tile first (last chunk, last tile), so the
    // grid still ends on light items and the CTAs resident at one time read one sequence's K/V
    if (p.kv_shard >= 0 || p.fused) {
      w.p = p.fused ? 0 : p.kv_shard;
    } else {
      q = udiv<FAST>(lin, p.f_cp);
      w.p = (int)(lin - q * (unsigned)p.cp);
      lin = q;
    }
    q = udiv<FAST>(lin, p.f_nslot);
    slot = (int)(lin - q * nslot);
    w.b = (int)q;
  }
  }
  const unsigned sq = udiv<FAST>((unsigned)slot, p.f_tpc);
  const int c = 2 * p.cp - 1 - (int)sq;
  const int j = p.TPC - 1 - (slot - (int)sq * p.TPC);
  const int q0 = p.cu_q[w.b];
  const int Tq = p.cu_q[w.b + 1] - q0;
  if (Tq <= 0) return w;
  const int cs = chunk_bound_f<FAST>(c, Tq, p), ce = chunk_bound_f<FAST>(c + 1, Tq, p);
  w.q_lo = cs + j * span;
  if (w.q_lo >= ce) return w;
  w.q_hi = min(w.q_lo + span, ce);
  if (p.q_shard >= 0 && shard_of_chunk(c, p.cp) != p.q_shard) return w;
  w.valid = 1;
  w.g = (int)udiv<FAST>((unsigned)w.h, p.f_G);
  w.q_row0 = q0 + w.q_lo;
  w.ntiles = 0;
  if (p.mode == CP_PASS_KV) {
    // kv tokens of the sequence (cached + new); the queries are its last Tq positions
    int kv0 = q0, Tkv = Tq;
    if (p.cu_kv != nullptr) {
      kv0 = p.cu_kv[w.b];
      Tkv = p.cu_kv[w.b + 1] - kv0;
    }
    const int C = Tkv - Tq;
    if (C < 0) {  // fewer kv tokens than new queries: flagged, the item is skipped
      report(p.err, CP_ERR_DEVICE_BOUNDS);
      w.valid = 0;
      return w;
    }
    w.qpos0 = C + w.q_lo;
    w.kv_row0 = kv0;
    if (p.fused) {  // the union of all shards' keys: positions [0, C + q_hi)
      w.ks[0] = 0;
      w.ke[0] = C + w.q_hi;
      w.nt[0] = (w.ke[0] + BN - 1) / BN;
      w.ks[1] = w.ke[1] = w.nt[1] = 0;
      w.ntiles = w.nt[0];
    } else {
#pragma unroll
      for (int i = 0; i < 2; ++i) {  // kv chunks s and 2cp-1-s, positions < C + q_hi
        const int ch = i == 0 ? w.p : 2 * p.cp - 1 - w.p;
        w.ks[i] = chunk_bound_f<FAST>(ch, Tkv, p);
        w.ke[i] = min(chunk_bound_f<FAST>(ch + 1, Tkv, p), C + w.q_hi);
        if (w.ke[i] < w.ks[i]) w.ke[i] = w.ks[i];
        w.nt[i] = (w.ke[i] - w.ks[i] + BN - 1) / BN;
        w.ntiles += w.nt[i];
      }
    }
  } else {
    const long long C = (long long)p.seq_lens_kv[w.b] - Tq;
    if (C < 0) {  // fewer kv tokens than new queries: flagged, the item is skipped
      report(p.err, CP_ERR_DEVICE_BOUNDS);
      w.valid = 0;
      return w;
    }
    w.qpos0 = C + w.q_lo;
    if (p.fused) {  // every rank's resident tokens any row can see, rank after rank
      w.n_local = 0;
      for (int r = w.r_lo; r < w.r_hi; ++r)
        w.ntiles += (rank_local_len(C + w.q_hi, r, p.cp, p.I) + BN - 1) / BN;
    } else {
      w.n_local = rank_local_len(C + w.q_hi, w.p, p.cp, p.I);
      w.ntiles = (w.n_local + BN - 1) / BN;
    }
  }
  return w;
}
CP_DEV Work decode_work(const TcParams& p, int hpc, int span = BM) {
  return decode_work_at(p, blockIdx.x, hpc, span);
}
// Fused pass-Q: this CTA's item, or (piece >= 0) one rank range of a split item.
template <bool FAST>
CP_DEV Work decode_split_work(const TcParams& p, int hpc, int span, int& piece) {
  unsigned lin = blockIdx.x;
  int r_lo = 0, r_hi = p.cp;
  piece = -1;
  if (p.split_k > 1 && lin >= (unsigned)p.n_whole) {
    piece = (int)(lin - (unsigned)p.n_whole);
    const int part = piece % p.split_k;
    lin = (unsigned)p.n_whole + (unsigned)(piece / p.split_k);
    r_lo = part * p.cp / p.split_k;
    r_hi = (part + 1) * p.cp / p.split_k;
  }
  return decode_work_at<FAST>(p, lin, hpc, span, r_lo, r_hi);
}

CP_DEV uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

CP_DEV void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// A warp's 32 staged rows (the boxes stage_rows_* wrote at sb) written out one row per store
// instruction: lane l carries columns [E l, E l + E), E = d / 32, so each warp-wide store covers
// a whole contiguous output row.  dst: row 0 of the warp; consecutive rows are `stride` elements
// apart.
template <int D>
CP_DEV void store_staged_f32(uint32_t sb, int lane, float* dst, long long stride) {
  constexpr int E = D / 32;
  const int col = E * lane, cin = col % 32;
  const uint32_t a0 = sb + (uint32_t)((col / 32) * 4096 + (cin % 4) * 4);
  const int chunk = cin / 4;
#pragma unroll 8
  for (int r = 0; r < 32; ++r) {
    const uint32_t a = a0 + (uint32_t)(r * 128) + ((uint32_t)(chunk ^ (r & 7)) << 4);
    float* g = dst + r * stride + col;
    if constexpr (E == 4) {
      float4 v;
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
      *reinterpret_cast<float4*>(g) = v;
    } else {
      float2 v;
      asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
      *reinterpret_cast<float2*>(g) = v;
    }
  }
}
template <int D>
CP_DEV void store_staged_bf16(uint32_t sb, int lane, __nv_bfloat16* dst, long long stride) {
  constexpr int E = D / 32;
  const int col = E * lane, cin = col % 64;
  const uint32_t a0 = sb + (uint32_t)((col / 64) * 4096 + (cin % 8) * 2);
  const int chunk = cin / 8;
#pragma unroll 8
  for (int r = 0; r < 32; ++r) {
    const uint32_t a = a0 + (uint32_t)(r * 128) + ((uint32_t)(chunk ^ (r & 7)) << 4);
    __nv_bfloat16* g = dst + r * stride + col;
    if constexpr (E == 4) {
      uint2 v;
      asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
      *reinterpret_cast<uint2*>(g) = v;
    } else {
      uint32_t v;
      asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
      *reinterpret_cast<uint32_t*>(g) = v;
    }
  }
}

CP_DEV void fail_timeout(volatile uint32_t* abort_flag, int32_t* err) {
  *abort_flag = 1u;
  report(err, CP_ERR_TIMEOUT);
}

// ---------------------------------------------------------------------------------- row softmax
// Packed two-lane fp32 arithmetic (f32x2 instructions of the sm_100 family) and 3-input max.
CP_DEV uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
CP_DEV void f2u(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
CP_DEV uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
CP_DEV uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
CP_DEV float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// The 128 scores of this thread's row (its TMEM lane), one TMEM round trip.
CP_DEV void load_row(uint32_t tS, float (&v0)[32], float (&v1)[32], float (&v2)[32],
                     float (&v3)[32]) {
  tmem_ld32(tS, v0);
  tmem_ld32(tS + 32, v1);
  tmem_ld32(tS + 64, v2);
  tmem_ld32(tS + 96, v3);
  tmem_wait_ld(v0);
  tmem_wait_ld(v1);
  tmem_wait_ld(v2);
  tmem_wait_ld(v3);
}

// Four independent packed partial sums keep the additions off one serial dependency chain.
CP_DEV void exp_chunk(float (&a)[32], uint64_t sc2, uint64_t n2, uint64_t& sum2) {
  uint64_t acc[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
  for (int k = 0; k < 32; k += 2) {
    float x0, x1;
    f2u(ffma2(f2(a[k], a[k + 1]), sc2, n2), x0, x1);
    a[k] = ex2(x0);
    a[k + 1] = ex2(x1);
    acc[(k >> 1) & 3] = fadd2(acc[(k >> 1) & 3], f2(a[k], a[k + 1]));
  }
  sum2 = fadd2(sum2, fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])));
}

// Row max of four 32-column chunks with four independent accumulators.
CP_DEV float max4x32(const float (&v0)[32], const float (&v1)[32], const float (&v2)[32],
                     const float (&v3)[32]) {
  float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
  for (int k = 0; k < 32; k += 2) {
    m0 = fmax3(m0, v0[k], v0[k + 1]);
    m1 = fmax3(m1, v1[k], v1[k + 1]);
    m2 = fmax3(m2, v2[k], v2[k + 1]);
    m3 = fmax3(m3, v3[k], v3[k + 1]);
  }
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// Online-softmax step of one row over a 128-key tile: columns > lim are masked (skipped when
// every row of the warp sees the whole tile), the running max m (log2 units) moves only when
// the tile max exceeds it by more than 2^8, and the scores become p = 2^(s*sc - m) in place.
// Returns alpha, the factor the row's O accumulator must be scaled by (l is updated here).
CP_DEV float row_softmax(float (&v0)[32], float (&v1)[32], float (&v2)[32], float (&v3)[32],
                         int lim, float sc, float& m, float& l) {
  if (!__all_sync(0xffffffffu, lim >= BN - 1)) {
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      v0[k] = k <= lim ? v0[k] : -INFINITY;
      v1[k] = k + 32 <= lim ? v1[k] : -INFINITY;
      v2[k] = k + 64 <= lim ? v2[k] : -INFINITY;
      v3[k] = k + 96 <= lim ? v3[k] : -INFINITY;
    }
  }
  const float m_tile = max4x32(v0, v1, v2, v3) * sc;
  float alpha = 1.f;
  if (m_tile > m + kRescaleThreshold) {  // first visible tile, or the max grew a lot
    alpha = ex2(m - m_tile);
    m = m_tile;
  }
  const float neg = (m == -INFINITY) ? 0.f : -m;
  const uint64_t sc2 = f2(sc, sc), n2 = f2(neg, neg);
  uint64_t sum2 = f2(0.f, 0.f);
  exp_chunk(v0, sc2, n2, sum2);
  exp_chunk(v1, sc2, n2, sum2);
  exp_chunk(v2, sc2, n2, sum2);
  exp_chunk(v3, sc2, n2, sum2);
  float s_lo, s_hi;
  f2u(sum2, s_lo, s_hi);
  l = l * alpha + (s_lo + s_hi);
  return alpha;
}

// Split form of row_softmax for kernels whose P buffer is already free when the scores
// arrive: mask + max + running-max update first (returns alpha) ...
CP_DEV float row_max_update(float (&v0)[32], float (&v1)[32], float (&v2)[32], float (&v3)[32],
                            int lim, float sc, float& m) {
  if (!__all_sync(0xffffffffu, lim >= BN - 1)) {
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      v0[k] = k <= lim ? v0[k] : -INFINITY;
      v1[k] = k + 32 <= lim ? v1[k] : -INFINITY;
      v2[k] = k + 64 <= lim ? v2[k] : -INFINITY;
      v3[k] = k + 96 <= lim ? v3[k] : -INFINITY;
    }
  }
  const float m_tile = max4x32(v0, v1, v2, v3) * sc;
  float alpha = 1.f;
  if (m_tile > m + kRescaleThreshold) {
    alpha = ex2(m - m_tile);
    m = m_tile;
  }
  return alpha;
}

// Exponentials of a row packed as bf16 pairs into the first 64 columns of its S buffer in TMEM
// (the A operand of a tensor-memory PV MMA), 16 columns per store; returns the row sum of p.
CP_DEV void exp_pack_tmem(float (&a)[32], uint64_t sc2, uint64_t n2, uint64_t& sum2, uint32_t taddr) {
  exp_chunk(a, sc2, n2, sum2);
  uint32_t pk[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) pk[k] = pack_bf16(a[2 * k], a[2 * k + 1]);
  tmem_st16(taddr, pk);
}
CP_DEV float row_exp_tmem(float (&v0)[32], float (&v1)[32], float (&v2)[32], float (&v3)[32],
                          float sc, float m, uint32_t tS) {
  const float neg = (m == -INFINITY) ? 0.f : -m;
  const uint64_t sc2 = f2(sc, sc), n2 = f2(neg, neg);
  uint64_t sum2 = f2(0.f, 0.f);
  exp_pack_tmem(v0, sc2, n2, sum2, tS);
  exp_pack_tmem(v1, sc2, n2, sum2, tS + 16);
  exp_pack_tmem(v2, sc2, n2, sum2, tS + 32);
  exp_pack_tmem(v3, sc2, n2, sum2, tS + 48);
  tmem_wait_st();
  float lo, hi;
  f2u(sum2, lo, hi);
  return lo + hi;
}

// P row (bf16) into a 128x128 P tile stored as two 64-column blocks in the 128-byte-swizzled
// K-major layout the MMA reads: 16-byte chunk c of row r sits at chunk c ^ (r % 8).
CP_DEV void store_p_row(uint32_t sP, int row, const float (&v0)[32], const float (&v1)[32],
                        const float (&v2)[32], const float (&v3)[32]) {
  const uint32_t prow = sP + row * 128;
  const uint32_t sw = (uint32_t)(row & 7);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float* a = c == 0 ? v0 : c == 1 ? v1 : c == 2 ? v2 : v3;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int col = c * 32 + h * 8;
      const uint32_t blk = (uint32_t)(col / 64), ch = (uint32_t)((col % 64) / 8);
      st_shared_v4(prow + blk * (BM * 128) + ((ch ^ sw) << 4), pack_bf16(a[h * 8], a[h * 8 + 1]),
                   pack_bf16(a[h * 8 + 2], a[h * 8 + 3]), pack_bf16(a[h * 8 + 4], a[h * 8 + 5]),
                   pack_bf16(a[h * 8 + 6], a[h * 8 + 7]));
    }
  }
}

// O row *= alpha in TMEM (warp-collective; nothing to do when no lane of the warp needs it).
template <int D>
CP_DEV void rescale_o(uint32_t tO, float alpha) {
  if (!__any_sync(0xffffffffu, alpha != 1.f)) return;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    float o[32];
    tmem_ld32(tO + c * 32, o);
    tmem_wait_ld(o);
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] *= alpha;
    tmem_st32(tO + c * 32, o);
  }
  tmem_wait_st();
}

// Final O row / l -> the partial output (f32) and its natural-log LSE (warp-collective).
template <int D>
CP_DEV void write_row(uint32_t tO, float m, float l, bool row_valid, float* dst, float* lse_dst) {
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    float o[32];
    tmem_ld32(tO + c * 32, o);
    tmem_wait_ld(o);
    if (row_valid && l > 0.f) {
#pragma unroll
      for (int k = 0; k < 32; k += 4)
        *reinterpret_cast<float4*>(dst + c * 32 + k) =
            make_float4(o[k] * inv_l, o[k + 1] * inv_l, o[k + 2] * inv_l, o[k + 3] * inv_l);
    }
  }
  if (row_valid) *lse_dst = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// Final O row / l -> bf16 output (round to nearest even) and its LSE (warp-collective).
template <int D>
CP_DEV void write_row_bf16(uint32_t tO, float m, float l, bool row_valid, __nv_bfloat16* dst,
                           float* lse_dst) {
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    float o[32];
    tmem_ld32(tO + c * 32, o);
    tmem_wait_ld(o);
    if (row_valid) {
#pragma unroll
      for (int k = 0; k < 32; k += 8)
        *reinterpret_cast<uint4*>(dst + c * 32 + k) = make_uint4(
            pack_bf16(o[k] * inv_l, o[k + 1] * inv_l), pack_bf16(o[k + 2] * inv_l, o[k + 3] * inv_l),
            pack_bf16(o[k + 4] * inv_l, o[k + 5] * inv_l), pack_bf16(o[k + 6] * inv_l, o[k + 7] * inv_l));
    }
  }
  if (row_valid) *lse_dst = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// Final O rows of one warp (its 32 TMEM lanes = 32 query rows, scaled by 1/l) staged in shared
// memory as 128-byte-swizzled boxes: f32 boxes of 32 columns x 32 rows (4 KB each, 16-byte chunk
// j of row r at chunk j ^ (r % 8)), or bf16 boxes of 64 columns.  A thread writes its own row,
// store_staged_* read them back a row per warp instruction; the swizzle keeps both directions
// free of bank conflicts.
template <int D>
CP_DEV void stage_rows_f32(uint32_t tO, float inv_l, uint32_t sbase, int lane) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    float o[32];
    tmem_ld32(tO + c * 32, o);
    tmem_wait_ld(o);
    const uint32_t rb = sbase + (uint32_t)(c * 4096 + lane * 128);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      st_shared_v4(rb + ((uint32_t)(j ^ (lane & 7)) << 4), __float_as_uint(o[4 * j] * inv_l),
                   __float_as_uint(o[4 * j + 1] * inv_l), __float_as_uint(o[4 * j + 2] * inv_l),
                   __float_as_uint(o[4 * j + 3] * inv_l));
  }
}
template <int D>
CP_DEV void stage_rows_bf16(uint32_t tO, float inv_l, uint32_t sbase, int lane) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    float o[32];
    tmem_ld32(tO + c * 32, o);
    tmem_wait_ld(o);
    const uint32_t rb = sbase + (uint32_t)((c >> 1) * 4096 + lane * 128);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      st_shared_v4(rb + ((uint32_t)(((c & 1) * 4 + j) ^ (lane & 7)) << 4),
                   pack_bf16(o[8 * j] * inv_l, o[8 * j + 1] * inv_l),
                   pack_bf16(o[8 * j + 2] * inv_l, o[8 * j + 3] * inv_l),
                   pack_bf16(o[8 * j + 4] * inv_l, o[8 * j + 5] * inv_l),
                   pack_bf16(o[8 * j + 6] * inv_l, o[8 * j + 7] * inv_l));
  }
}

// ---------------------------------------------------------------------------------- kernel
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc1_kernel(const __grid_constant__ CUtensorMap map_q,
                      const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v, const TcParams p) {
  using Ly = Layout<D>;
  constexpr int KB = D / 64;  // 64-column (128-byte) blocks of a head row
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Work w = decode_work(p, 1);
  if (!w.valid) return;  // uniform over the CTA

  if (w.ntiles == 0) {  // no visible key in this pair: an empty partial
    if (warp >= 2) {
      const int row = (warp & 3) * 32 + lane;
      if (w.q_lo + row < w.q_hi)
        p.lse[((long long)w.p * p.Nq + w.q_row0 + row) * p.Hq + w.h] = -INFINITY;
    }
    return;
  }

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const uint32_t sQ = base + Ly::oQ, sK = base + Ly::oK, sV = base + Ly::oV, sP = base + Ly::oP;
  const uint32_t bars = base + Ly::oBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(sbase + Ly::oMisc);
  volatile uint32_t* abort_flag = misc + 1;

  if (threadIdx.x == 0) {
    mbar_init(bar(Ly::bQ), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(Ly::bKF + s), 1);
      mbar_init(bar(Ly::bVF + s), 1);
      mbar_init(bar(Ly::bKE + s), 1);
      mbar_init(bar(Ly::bVE + s), 1);
    }
    mbar_init(bar(Ly::bS), 1);
    mbar_init(bar(Ly::bS + 1), 1);
    mbar_init(bar(Ly::bP), 4);
    mbar_init(bar(Ly::bO), 1);
    mbar_init(bar(Ly::bDone), 1);
    misc[1] = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(misc), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const uint32_t tO = tmem + 256;  // S buffers at columns [0,128) and [128,256)

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      mbar_expect_tx(bar(Ly::bQ), Ly::kQ);
#pragma unroll
      for (int kb = 0; kb < KB; ++kb)
        tma_load_2d(sQ + kb * BM * 128, &map_q, w.h * D + kb * 64, w.q_row0, bar(Ly::bQ));
      int lk0 = -1, lk1 = -1, lv0 = -1, lv1 = -1;  // phase of the last K / V fill per stage
      const int32_t* trow =
          p.mode == CP_PASS_Q ? p.tables + ((long long)w.p * p.B + w.b) * p.max_blocks : nullptr;
      int pid[BN / 16];  // pass-Q: page ids of the next tile, loaded one tile ahead
      if (p.mode == CP_PASS_Q) fetch_page_ids(trow, 0, w.n_local, p.max_blocks, pid);
      bool ok = true;
      for (int t = 0; t < w.ntiles; ++t) {
        const int s = t % NS;
        const uint32_t ph = (uint32_t)(t / NS) & 1u;
        if (!mbar_wait(bar(Ly::bKE + s), ph ^ 1u, abort_flag, p.budget)) { ok = false; break; }
        const uint32_t dK = sK + s * Ly::kKV, dV = sV + s * Ly::kKV;
        if (p.mode == CP_PASS_KV) {
          const bool r0 = t < w.nt[0];
          const int y = w.kv_row0 + (r0 ? w.ks[0] + t * BN : w.ks[1] + (t - w.nt[0]) * BN);
          mbar_expect_tx(bar(Ly::bKF + s), Ly::kKV);
#pragma unroll
          for (int kb = 0; kb < KB; ++kb)
            tma_load_2d(dK + kb * BN * 128, &map_k, w.g * D + kb * 64, y, bar(Ly::bKF + s));
          if (!mbar_wait(bar(Ly::bVE + s), ph ^ 1u, abort_flag, p.budget)) { ok = false; break; }
          if (p.debug & 1) {  // testing: V never arrives, the consumer's wait expires
            if (s == 0) lk0 = (int)ph; else lk1 = (int)ph;
            continue;
          }
          mbar_expect_tx(bar(Ly::bVF + s), Ly::kKV);
#pragma unroll
          for (int kb = 0; kb < KB; ++kb)
            tma_load_2d(dV + kb * BN * 128, &map_v, w.g * D + kb * 64, y, bar(Ly::bVF + s));
        } else {
          int rows[BN / 16];
          page_rows(pid, t, w.n_local, p.pool, p.Hkv, w.p, w.g, p.err, rows);
          if (t + 1 < w.ntiles) fetch_page_ids(trow, t + 1, w.n_local, p.max_blocks, pid);
          mbar_expect_tx(bar(Ly::bKF + s), Ly::kKV);
#pragma unroll
          for (int i = 0; i < BN / 16; ++i)
#pragma unroll
            for (int kb = 0; kb < KB; ++kb)
              tma_load_2d(dK + kb * BN * 128 + i * 16 * 128, &map_k, kb * 64, rows[i],
                          bar(Ly::bKF + s));
          if (!mbar_wait(bar(Ly::bVE + s), ph ^ 1u, abort_flag, p.budget)) { ok = false; break; }
          if (p.debug & 1) {
            if (s == 0) lk0 = (int)ph; else lk1 = (int)ph;
            continue;
          }
          mbar_expect_tx(bar(Ly::bVF + s), Ly::kKV);
#pragma unroll
          for (int i = 0; i < BN / 16; ++i)
#pragma unroll
            for (int kb = 0; kb < KB; ++kb)
              tma_load_2d(dV + kb * BN * 128 + i * 16 * 128, &map_v, kb * 64, rows[i],
                          bar(Ly::bVF + s));
        }
        if (s == 0) lk0 = (int)ph; else lk1 = (int)ph;
        if (s == 0) lv0 = (int)ph; else lv1 = (int)ph;
      }
      if (!ok) fail_timeout(abort_flag, p.err);
      // drain: every copy issued into this CTA's shared memory has landed before it exits
      mbar_wait(bar(Ly::bQ), 0u, nullptr, p.budget);
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        const int lk = s == 0 ? lk0 : lk1, lv = s == 0 ? lv0 : lv1;
        if (lk >= 0) mbar_wait(bar(Ly::bKF + s), (uint32_t)lk, nullptr, p.budget);
        if (lv >= 0) mbar_wait(bar(Ly::bVF + s), (uint32_t)lv, nullptr, p.budget);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16_f32(BM, BN, false, false);
      const uint32_t id_pv = idesc_bf16_f32(BM, D, false, true);
      auto issue_qk = [&](int t) {
        const uint32_t kst = sK + (t % NS) * Ly::kKV;
        const uint32_t dS = tmem + (uint32_t)((t & 1) * BN);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * (BM * 128) + (k % 4) * 32;
          const uint32_t offk = (k / 4) * (BN * 128) + (k % 4) * 32;
          mma_ss(dS, desc_sw128(sQ + off, 16, 1024), desc_sw128(kst + offk, 16, 1024), id_qk,
                 k > 0 ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(bar(Ly::bQ), 0u, abort_flag, p.budget);
      if (ok) ok = mbar_wait(bar(Ly::bKF), 0u, abort_flag, p.budget);
      if (ok) {
        tc_fence_after();
        issue_qk(0);
        mma_commit(bar(Ly::bS));
        mma_commit(bar(Ly::bKE));
      }
      for (int t = 0; ok && t < w.ntiles; ++t) {
        if (t + 1 < w.ntiles) {
          const int s1 = (t + 1) % NS;
          ok = mbar_wait(bar(Ly::bKF + s1), (uint32_t)((t + 1) / NS) & 1u, abort_flag, p.budget);
          if (!ok) break;
          tc_fence_after();
          issue_qk(t + 1);
          mma_commit(bar(Ly::bS + ((t + 1) & 1)));
          mma_commit(bar(Ly::bKE + s1));
        }
        ok = mbar_wait(bar(Ly::bP), (uint32_t)t & 1u, abort_flag, p.budget);
        if (!ok) break;
        const int s = t % NS;
        ok = mbar_wait(bar(Ly::bVF + s), (uint32_t)(t / NS) & 1u, abort_flag, p.budget);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vst = sV + s * Ly::kKV;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint32_t offp = (k / 4) * (BM * 128) + (k % 4) * 32;
          mma_ss(tO, desc_sw128(sP + offp, 16, 1024), desc_sw128(vst + k * 16 * 128, BN * 128, 1024),
                 id_pv, (t > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(bar(Ly::bO));
        mma_commit(bar(Ly::bVE + s));
      }
      if (!ok) fail_timeout(abort_flag, p.err);
      // every MMA issued by this thread has retired before TMEM is released
      mma_commit(bar(Ly::bDone));
      mbar_wait(bar(Ly::bDone), 0u, nullptr, p.budget);
    }
  } else {
    // ------------------------------------------------------------------ softmax warpgroup
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const bool row_valid = w.q_lo + row < w.q_hi;
    const long long qpos = w.qpos0 + row;
    // keys visible to this row within the pass-Q range (local indices < nvis)
    int nvis = 0;
    if (p.mode == CP_PASS_Q) nvis = min(w.n_local, rank_local_len(qpos + 1, w.p, p.cp, p.I));
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < w.ntiles; ++t) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(Ly::bS + (t & 1)), (uint32_t)(t >> 1) & 1u, abort_flag, p.budget));
      if (!ok) break;
      tc_fence_after();
      float s0[32], s1[32], s2[32], s3[32];
      load_row(tmem + lane_off + (uint32_t)((t & 1) * BN), s0, s1, s2, s3);
      // last visible key column of this row in the tile (all keys <= lim are visible)
      int lim;
      if (p.mode == CP_PASS_KV) {
        const bool r0 = t < w.nt[0];
        const int k0 = r0 ? w.ks[0] + t * BN : w.ks[1] + (t - w.nt[0]) * BN;
        const int ke = r0 ? w.ke[0] : w.ke[1];
        lim = (int)min((long long)ke - 1, qpos) - k0;
      } else {
        lim = nvis - 1 - t * BN;
      }
      const float alpha = row_softmax(s0, s1, s2, s3, lim, p.scale_log2, m, l);
      if (t > 0) {  // PV(t-1) has finished: the P buffer is free and O is stable
        ok = __all_sync(0xffffffffu, mbar_wait(bar(Ly::bO), (uint32_t)(t - 1) & 1u, abort_flag, p.budget));
        if (!ok) break;
        tc_fence_after();
        rescale_o<D>(tO + lane_off, alpha);
      }
      store_p_row(sP, row, s0, s1, s2, s3);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Ly::bP));
    }
    if (ok)
      ok = __all_sync(0xffffffffu, mbar_wait(bar(Ly::bO), (uint32_t)(w.ntiles - 1) & 1u,
                                             abort_flag, p.budget));
    if (ok) {
      tc_fence_after();
      if (p.fused) {
        const long long frow = (long long)(w.q_row0 + row) * p.Hq + w.h;
        write_row_bf16<D>(tO + lane_off, m, l, row_valid, p.out_final + frow * D, p.lse_final + frow);
      } else {
        const long long orow = ((long long)w.p * p.Nq + w.q_row0 + row) * p.Hq + w.h;
        write_row<D>(tO + lane_off, m, l, row_valid, p.out + orow * D, p.lse + orow);
      }
    } else {
      fail_timeout(abort_flag, p.err);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------------- kernel 2
// Two query tiles per CTA sharing every K/V tile: tiles 0 and 1 are heads h, h+1 of one kv group
// over the same 128 rows (even G), or two consecutive 128-row tiles of one head.  Warps: 0 TMA
// producer, 1 TMEM owner + MMA issuer, 2-3 idle, 4-7 softmax of tile 0, 8-11 softmax of tile 1
// (warp w reads TMEM lanes 32 (w % 4) ..).  Three aligned warpgroups put one warp of each on
// every SM sub-partition, so the register budgets (setmaxnreg) can differ by role: 88 for the
// producer / MMA warpgroup and 208 for each softmax warpgroup, 88 + 2 x 208 = 504 = 3 x the 168
// a thread of the 384-thread launch gets.  (With 320 threads two sub-partitions host three warps
// and 168 is the ceiling for every warp; the softmax row then spills.  Measured: 208 / 88 runs
// the full and long prefill partials 4% faster than 168 for all; 224 / 56 starves the MMA
// issuer and is 2-6% slower.)  TMEM: S0 [0,128), S1 [128,256), O0 [256, 256+D),
// O1 [256+D, 256+2D).  The softmax writes P as packed bf16 pairs over the first 64 columns of its
// own S buffer and the PV MMA reads A from tensor memory.  K and V tiles stream through a 4-slot
// ring (load i: K(t) for i = 2t, V(t) for i = 2t+1; 4 slots measured ~1.5% faster than 5).
// Tensor-core order per key tile t:
//   PV0(t) | QK0(t+1) | PV1(t) | QK1(t+1)
// so the softmax of each tile overlaps the other tile's two MMAs.
constexpr int kThreads2 = 384;
constexpr int kReg2Producer = 88, kReg2Softmax = 208;
static_assert(kReg2Producer + 2 * kReg2Softmax <= 3 * 168, "register budgets exceed the launch");

template <int D>
struct Layout2 {
  static constexpr int NSLOT = 4;
  static constexpr int kQ = BM * D * 2;
  static constexpr int kKV = BN * D * 2;
  static constexpr int oQ = 0;
  static constexpr int oKV = 2 * kQ;
  static constexpr int oBar = oKV + NSLOT * kKV;
  static constexpr int bQ = 0, bFull = 1, bEmpty = bFull + NSLOT, bS = bEmpty + NSLOT, bP = bS + 2,
                       bO = bP + 2, bDone = bO + 2, nBar = bDone + 1;
  static constexpr int oMisc = oBar + nBar * 8;
  static constexpr int kBytes = oMisc + 16;
  static constexpr int kAlloc = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
  static_assert(kAlloc <= 232448, "dynamic shared memory beyond the 227 KB per-CTA limit");
};

// PG: paged K/V as whole-page boxes (pass-Q, d = 128).  TT: the two "tiles" of the CTA are two
// consecutive 128-row query tiles of one head (any G) instead of two heads of a kv group (even G).
// FQ: fused pass-Q, the item walks every rank's resident pages (rank after rank).
template <int D, bool PG, bool TT, bool FQ>
__global__ void __launch_bounds__(kThreads2, 1)
    prefill_tc2_kernel(const __grid_constant__ CUtensorMap map_q,
                       const __grid_constant__ CUtensorMap map_k,
                       const __grid_constant__ CUtensorMap map_v,
                       const TcParams p) {
  using Ly = Layout2<D>;
  constexpr int NSLOT = Ly::NSLOT;
  constexpr int KB = D / 64;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int piece = -1;  // fused pass-Q: >= 0 when this CTA runs one rank range of a split item
  const Work w = FQ ? decode_split_work<false>(p, TT ? 1 : 2, TT ? 2 * BM : BM, piece)
                    : (TT ? decode_work(p, 1, 2 * BM) : decode_work(p, 2));
  if (!w.valid) return;

  if (w.ntiles == 0) {  // empty pair
    if (warp >= 4) {
      const int tile = (warp - 4) >> 2;
      const int row = (warp & 3) * 32 + lane + (TT ? tile * BM : 0);  // within the item
      const int hcol = w.h + (TT ? 0 : tile);
      if (w.q_lo + row < w.q_hi) {
        if (piece >= 0) {  // no visible key in this rank range
          p.ws_lse[((long long)piece * 2 + tile) * BM + (warp & 3) * 32 + lane] = -INFINITY;
        } else if (p.fused) {  // no visible key at all: exact attention is 0 with lse -inf
          const long long frow = (long long)(w.q_row0 + row) * p.Hq + hcol;
          for (int c = 0; c < D; ++c) p.out_final[frow * D + c] = __float2bfloat16_rn(0.f);
          p.lse_final[frow] = -INFINITY;
        } else {
          p.lse[((long long)w.p * p.Nq + w.q_row0 + row) * p.Hq + hcol] = -INFINITY;
        }
      }
    }
    return;
  }

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const uint32_t sQ = base + Ly::oQ, sKV = base + Ly::oKV;
  const uint32_t bars = base + Ly::oBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(sbase + Ly::oMisc);
  volatile uint32_t* abort_flag = misc + 1;

  if (threadIdx.x == 0) {
    mbar_init(bar(Ly::bQ), 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(bar(Ly::bFull + s), 1);
      mbar_init(bar(Ly::bEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(Ly::bS + i), 1);
      mbar_init(bar(Ly::bP + i), 4);
      mbar_init(bar(Ly::bO + i), 1);
    }
    mbar_init(bar(Ly::bDone), 1);
    misc[1] = 0u;
    fence_mbar_init();
    // the Q tiles of both heads load while the CTA is still setting up (TMEM, barriers)
    tma_prefetch_desc(&map_q);
    mbar_expect_tx(bar(Ly::bQ), 2 * Ly::kQ);
#pragma unroll
    for (int i = 0; i < 2; ++i)  // two heads at the tile's rows, or one head's two row tiles
#pragma unroll
      for (int kb = 0; kb < KB; ++kb)
        tma_load_2d(sQ + i * Ly::kQ + kb * BM * 128, &map_q, (w.h + (TT ? 0 : i)) * D + kb * 64,
                    w.q_row0 + (TT ? i * BM : 0), bar(Ly::bQ));
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(misc), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  // each budget change sits at the head of its warpgroup's branch, so the code of a role is
  // compiled under that role's budget
  if (warp < 4) {
  regs_dec<kReg2Producer>();
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      int lastph[NSLOT];  // parity of the last fill of each slot (-1: never filled)
#pragma unroll
      for (int i = 0; i < NSLOT; ++i) lastph[i] = -1;
      int prow[BN / 16];  // pass-Q: element rows of the current tile's pages (K and V alike)
      int pid[BN / 16];   // pass-Q: page ids of the next tile, loaded one tile ahead
      auto table_of = [&](int r) { return p.tables + ((long long)r * p.B + w.b) * p.max_blocks; };
      const int32_t* trow = p.mode == CP_PASS_Q ? table_of(w.p) : nullptr;
      // fused pass-Q: the key tiles walk rank 0, 1, .. in turn (FQ only)
      const long long kv_end = w.qpos0 - w.q_lo + w.q_hi;
      RankWalk kw{0, 0, 0, 0};
      if constexpr (FQ) {
        kw = walk_start(kv_end, p.cp, p.I, w.r_lo, w.r_hi);
        fetch_page_ids(table_of(kw.r), kw.tr, kw.n_r, p.max_blocks, pid);
      } else {
        if (p.mode == CP_PASS_Q) fetch_page_ids(trow, 0, w.n_local, p.max_blocks, pid);
      }
      bool ok = true;
      for (int i = 0; i < 2 * w.ntiles; ++i) {
        const int slot = i % NSLOT;
        const uint32_t ph = (uint32_t)(i / NSLOT) & 1u;
        const int t = i >> 1;
        const bool isV = (i & 1) != 0;
        if (!mbar_wait(bar(Ly::bEmpty + slot), ph ^ 1u, abort_flag, p.budget)) { ok = false; break; }
        if (isV && (p.debug & 1)) continue;  // testing: V never arrives
        const uint32_t dst = sKV + slot * Ly::kKV;
        const CUtensorMap* map = isV ? &map_v : &map_k;
        mbar_expect_tx(bar(Ly::bFull + slot), Ly::kKV);
        if (p.mode == CP_PASS_KV) {
          const bool r0 = t < w.nt[0];
          const int y = w.kv_row0 + (r0 ? w.ks[0] + t * BN : w.ks[1] + (t - w.nt[0]) * BN);
#pragma unroll
          for (int kb = 0; kb < KB; ++kb)
            tma_load_2d(dst + kb * BN * 128, map, w.g * D + kb * 64, y, bar(Ly::bFull + slot));
        } else {
          if (!isV) {  // page rows of tile t (reused for its V load)
            if constexpr (FQ) {
              page_rows(pid, kw.tr, kw.n_r, p.pool, p.Hkv, kw.r, w.g, p.err, prow);
              RankWalk kn = kw;  // the next tile
              walk_next(kn, kv_end, p.cp, p.I, w.r_hi);
              if (t + 1 < w.ntiles) fetch_page_ids(table_of(kn.r), kn.tr, kn.n_r, p.max_blocks, pid);
              kw = kn;
            } else {
              page_rows(pid, t, w.n_local, p.pool, p.Hkv, w.p, w.g, p.err, prow);
              if (t + 1 < w.ntiles) fetch_page_ids(trow, t + 1, w.n_local, p.max_blocks, pid);
            }
          }
          if constexpr (PG) {
#pragma unroll
            for (int j = 0; j < BN / 16; ++j)
              tma_load_4d(dst + j * 4096, map, 0, 0, 0, prow[j] >> 3, bar(Ly::bFull + slot));
          } else {
#pragma unroll
            for (int j = 0; j < BN / 16; ++j)
#pragma unroll
              for (int kb = 0; kb < KB; ++kb)
                tma_load_2d(dst + kb * BN * 128 + j * 16 * 128, map, kb * 64, prow[j],
                            bar(Ly::bFull + slot));
          }
        }
#pragma unroll
        for (int k = 0; k < NSLOT; ++k)
          if (k == slot) lastph[k] = (int)ph;
      }
      if (!ok) fail_timeout(abort_flag, p.err);
      mbar_wait(bar(Ly::bQ), 0u, nullptr, p.budget);
#pragma unroll
      for (int k = 0; k < NSLOT; ++k)
        if (lastph[k] >= 0) mbar_wait(bar(Ly::bFull + k), (uint32_t)lastph[k], nullptr, p.budget);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16_f32(BM, BN, false, false);
      const uint32_t id_pv = idesc_bf16_f32(BM, D, false, true);
      // shared-memory descriptors built once (Q tiles, ring slot 0 as a K and as a V operand) and
      // advanced by constant offsets: the issuing thread sits on the critical path between a
      // softmax hand-off and the tensor pipe, so its instructions per MMA matter
      const uint64_t dq0 = desc_sw128(sQ, 16, 1024);
      const uint64_t dk0 = desc_sw128(sKV, 16, PG ? 2048u : 1024u);
      const uint64_t dv0 = PG ? desc_sw128(sKV, 1024, 2048) : desc_sw128(sKV, BN * 128, 1024);
      auto issue_qk = [&](int tile, int slot) {
        const uint64_t dq = desc_advance(dq0, (uint32_t)(tile * Ly::kQ));
        const uint64_t dk = desc_advance(dk0, (uint32_t)(slot * Ly::kKV));
        const uint32_t dS = tmem + (uint32_t)(tile * BN);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offq = (kk / 4) * (BM * 128) + (kk % 4) * 32;
          // paged slot: 64-column block at +1 KB, 8-key groups 2 KB apart; tiled: block at
          // +BN x 128 B, groups 1 KB apart
          const uint32_t offk = (kk / 4) * (PG ? 1024u : (uint32_t)(BN * 128)) + (kk % 4) * 32;
          mma_ss(dS, desc_advance(dq, offq), desc_advance(dk, offk), id_qk, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int tile, int slot, bool acc) {
        const uint64_t dv = desc_advance(dv0, (uint32_t)(slot * Ly::kKV));
        const uint32_t dO = tmem + 256u + (uint32_t)(tile * D);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // 16 keys = one page: paged slot (halves 1 KB apart, 8-key groups 2 KB apart) or
          // the tiled layout (halves BN x 128 B apart, groups 1 KB apart)
          const uint64_t bd = desc_advance(dv, PG ? kk * 4096u : kk * 16u * 128u);
          // P: 8 packed TMEM columns per 16 keys, the A operand from tensor memory
          mma_ts(dO, tmem + (uint32_t)(tile * BN + kk * 8), bd, id_pv, (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(bar(Ly::bQ), 0u, abort_flag, p.budget);
      if (ok) ok = mbar_wait(bar(Ly::bFull + 0), 0u, abort_flag, p.budget);  // K(0): load 0
      if (ok) {
        tc_fence_after();
        issue_qk(0, 0);
        mma_commit(bar(Ly::bS + 0));
        issue_qk(1, 0);
        mma_commit(bar(Ly::bS + 1));
        mma_commit(bar(Ly::bEmpty + 0));
      }
      for (int t = 0; ok && t < w.ntiles; ++t) {
        const int iv = 2 * t + 1, ik = 2 * t + 2;
        const int sv = iv % NSLOT, sk = ik % NSLOT;
        ok = mbar_wait(bar(Ly::bFull + sv), (uint32_t)(iv / NSLOT) & 1u, abort_flag, p.budget);
        if (!ok) break;
        ok = mbar_wait(bar(Ly::bP + 0), (uint32_t)t & 1u, abort_flag, p.budget);
        if (!ok) break;
        tc_fence_after();
        issue_pv(0, sv, t > 0);
        mma_commit(bar(Ly::bO + 0));
        const bool more = t + 1 < w.ntiles;
        if (more) {
          ok = mbar_wait(bar(Ly::bFull + sk), (uint32_t)(ik / NSLOT) & 1u, abort_flag, p.budget);
          if (!ok) break;
          tc_fence_after();
          issue_qk(0, sk);
          mma_commit(bar(Ly::bS + 0));
        }
        ok = mbar_wait(bar(Ly::bP + 1), (uint32_t)t & 1u, abort_flag, p.budget);
        if (!ok) break;
        tc_fence_after();
        issue_pv(1, sv, t > 0);
        mma_commit(bar(Ly::bO + 1));
        mma_commit(bar(Ly::bEmpty + sv));
        if (more) {
          issue_qk(1, sk);
          mma_commit(bar(Ly::bS + 1));
          mma_commit(bar(Ly::bEmpty + sk));
        }
      }
      if (!ok) fail_timeout(abort_flag, p.err);
      mma_commit(bar(Ly::bDone));
      mbar_wait(bar(Ly::bDone), 0u, nullptr, p.budget);
    }
  }
  } else {
    regs_inc<kReg2Softmax>();
    // ------------------------------------------------------------------ softmax, one WG per tile
    const int tile = (warp - 4) >> 2;
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const int rofs = TT ? tile * BM : 0;   // this tile's first row within the item
    const int hcol = w.h + (TT ? 0 : tile);  // this tile's query head
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_off + (uint32_t)(tile * BN);
    const uint32_t tO = tmem + lane_off + 256u + (uint32_t)(tile * D);
    const bool row_valid = w.q_lo + rofs + row < w.q_hi;
    const long long qpos = w.qpos0 + rofs + row;
    int nvis = 0;
    constexpr bool walk = FQ;  // fused pass-Q: rank after rank
    const long long kv_end = w.qpos0 - w.q_lo + w.q_hi;
    const uint32_t g_rr = (long long)p.I * p.cp < (1ll << 31) ? (uint32_t)(p.I * p.cp) : (1u << 31);
    RankWalk kw{0, 0, 0, 0};
    if constexpr (walk) {
      kw = walk_start(kv_end, p.cp, p.I, w.r_lo, w.r_hi);
      nvis = min(kw.n_r, rank_len32(qpos + 1, kw.r, p.I, g_rr));
    } else {
      if (p.mode == CP_PASS_Q) nvis = min(w.n_local, rank_local_len(qpos + 1, w.p, p.cp, p.I));
    }
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < w.ntiles; ++t) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(Ly::bS + tile), (uint32_t)t & 1u, abort_flag, p.budget));
      if (!ok) break;
      tc_fence_after();
      float s0[32], s1[32], s2[32], s3[32];
      load_row(tS, s0, s1, s2, s3);
      int lim;
      if (p.mode == CP_PASS_KV) {
        const bool r0 = t < w.nt[0];
        const int k0 = r0 ? w.ks[0] + t * BN : w.ks[1] + (t - w.nt[0]) * BN;
        const int ke = r0 ? w.ke[0] : w.ke[1];
        lim = (int)min((long long)ke - 1, qpos) - k0;
      } else if constexpr (!walk) {
        lim = nvis - 1 - t * BN;
      } else {
        if (kw.tr == 0 && t > 0) nvis = min(kw.n_r, rank_len32(qpos + 1, kw.r, p.I, g_rr));
        lim = nvis - 1 - kw.tr * BN;
        walk_next(kw, kv_end, p.cp, p.I, w.r_hi);
      }
      const float alpha = row_max_update(s0, s1, s2, s3, lim, p.scale_log2, m);
      // S(t) complete implies PV(t-1) complete (it was issued before QK(t)): O is stable and
      // the S columns may take P(t)
      l = l * alpha + row_exp_tmem(s0, s1, s2, s3, p.scale_log2, m, tS);
      if (t > 0) rescale_o<D>(tO, alpha);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Ly::bP + tile));
    }
    if (ok)
      ok = __all_sync(0xffffffffu, mbar_wait(bar(Ly::bO + tile), (uint32_t)(w.ntiles - 1) & 1u,
                                             abort_flag, p.budget));
    // every load and MMA of the item is done: a kernel launched after this one (the merge)
    // may be scheduled once all CTAs are here
    griddep_launch_dependents();
    if (ok) {
      tc_fence_after();
      const long long frow = (long long)(w.q_row0 + rofs + row) * p.Hq + hcol;
      const long long orow = ((long long)w.p * p.Nq + w.q_row0 + rofs + row) * p.Hq + hcol;
      if (piece >= 0) {  // one rank range of a split item: its partial for the merge kernel
        // the workspace holds all 32 rows of every warp (rows past the item and rows that saw
        // no key are written as well, and never read), so they always go out as whole rows
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const uint32_t sb = (tile == 0 ? sQ : sKV) + (uint32_t)(q4 * 32 * D * 4);
        stage_rows_f32<D>(tO, inv_l, sb, lane);
        __syncwarp();
        const long long wrow0 = ((long long)piece * 2 + tile) * BM + q4 * 32;
        store_staged_f32<D>(sb, lane, p.ws_out + wrow0 * D, D);
        if (row_valid) p.ws_lse[wrow0 + lane] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      } else if (p.row_out && w.q_lo + rofs + q4 * 32 + 32 <= w.q_hi) {
        // all 32 rows of this warp are real: stage them in shared memory (128-byte-swizzled
        // boxes, conflict-free both ways) and read them back so that each warp-wide store
        // writes one whole contiguous output row.  Head 0 stages in the Q tiles (free: its last
        // PV completed after the other head's last QK), head 1 in the K/V ring (free: its last
        // PV is the CTA's last MMA).  Measured against TMA tensor stores of the same boxes: the
        // stores' reads of the staging buffer took ~1.15 us per warp before the CTA could exit;
        // full partials 0.211 -> 0.207 ms, long 5.64 -> 5.51 ms.
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const uint32_t sb = (tile == 0 ? sQ : sKV) + (uint32_t)(q4 * 32 * D * (p.fused ? 2 : 4));
        if (p.fused) stage_rows_bf16<D>(tO, inv_l, sb, lane);
        else stage_rows_f32<D>(tO, inv_l, sb, lane);
        __syncwarp();
        const long long z = (p.fused ? 0 : (long long)w.p * p.Nq) + w.q_row0 + rofs + q4 * 32;
        if (p.fused)
          store_staged_bf16<D>(sb, lane, p.out_final + (z * p.Hq + hcol) * D, (long long)p.Hq * D);
        else
          store_staged_f32<D>(sb, lane, p.out + (z * p.Hq + hcol) * D, (long long)p.Hq * D);
        const float lse_v = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        if (p.fused) p.lse_final[frow] = lse_v;
        else p.lse[orow] = lse_v;
      } else if (p.fused) {
        write_row_bf16<D>(tO, m, l, row_valid, p.out_final + frow * D, p.lse_final + frow);
      } else {
        write_row<D>(tO, m, l, row_valid, p.out + orow * D, p.lse + orow);
      }
    } else {
      fail_timeout(abort_flag, p.err);
    }
    }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Fused pass-Q, split tail: the split_k rank-range partials of each split item (normalised rows
// and natural-log LSEs, written by the pieces above) combined as cp_lse_merge does -- weights
// exp(lse_k - max), a range with lse = -inf contributes nothing -- into the item's bf16 output
// rows and LSEs.  One CTA per split item, one warp per (tile, row).  Launched as a programmatic
// dependent of the attention kernel.
template <int D, bool TT>
__global__ void __launch_bounds__(256) fq_split_merge_kernel(const TcParams p) {
  constexpr int E = D / 32;  // values per lane
  griddep_wait();
  const Work w = decode_work_at<false>(p, (unsigned)p.n_whole + blockIdx.x, TT ? 1 : 2, TT ? 2 * BM : BM);
  if (!w.valid) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int u = warp; u < 2 * BM; u += 8) {
    const int tile = u / BM, row = u % BM;
    const int rofs = TT ? tile * BM : 0;
    if (w.q_lo + rofs + row >= w.q_hi) continue;
    const int hcol = w.h + (TT ? 0 : tile);
    float M = -INFINITY;
    for (int k = 0; k < p.split_k; ++k) {
      const long long wrow = (((long long)blockIdx.x * p.split_k + k) * 2 + tile) * BM + row;
      M = fmaxf(M, p.ws_lse[wrow] * kLog2e);
    }
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    if (M > -INFINITY) {
      for (int k = 0; k < p.split_k; ++k) {
        const long long wrow = (((long long)blockIdx.x * p.split_k + k) * 2 + tile) * BM + row;
        const float lk = p.ws_lse[wrow] * kLog2e;
        if (!(lk > -INFINITY)) continue;  // an empty range's rows were never written
        const float wk = exp2f(lk - M);
        wsum += wk;
        const float* src = p.ws_out + wrow * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += wk * src[e];
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const long long frow = (long long)(w.q_row0 + rofs + row) * p.Hq + hcol;
    __nv_bfloat16* dst = p.out_final + frow * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2)
      *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
    if (lane == 0) p.lse_final[frow] = wsum > 0.f ? (M + log2f(wsum)) * kLn2 : -INFINITY;
  }
}

// ---------------------------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2D bf16 tensor map over `rows` rows of `cols` elements (row pitch `pitch_elems`), box of
// 64 columns x box_rows rows, 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* m, const void* base, unsigned long long cols, unsigned long long rows,
              unsigned long long pitch_elems, unsigned box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_elems * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Fused pass-Q work items cost about the same (every row sees its ranks' whole cached context),
// so a grid of n items on S SMs (one CTA each) takes ceil(n / S) item times.  When the last wave
// is partly empty, its rem = n mod S items are each cut into k rank ranges (k <= cp; ranks hold
// equal shares, so a piece of at most ceil(cp / k) ranks costs that many cp-ths of an item) whose
// partials fq_split_merge_kernel combines: the tail then takes ceil(rem k / S) ceil(cp / k) / cp
// item times.  The smallest k with the shortest tail is taken, and only when it saves at least a
// quarter of an item (each piece repeats an item's prologue and epilogue).
struct SplitPlan {
  long long n_split;  // items run as pieces (the last n_split items of the grid)
  int k;              // pieces per split item; 1 = no split
};
SplitPlan split_plan(long long items, int cp, int sms) {
  SplitPlan sp{0, 1};
  if (sms <= 0 || cp < 2 || items <= 0) return sp;
  const long long rem = items % sms;
  if (rem == 0) return sp;
  double best = 1.0;
  int bk = 1;
  for (int k = 2; k <= cp; ++k) {
    const double t = (double)((rem * k + sms - 1) / sms) * ((cp + k - 1) / k) / cp;
    if (t < best - 1e-9) {
      best = t;
      bk = k;
    }
  }
  if (best > 0.75) return sp;
  sp.n_split = rem;
  sp.k = bk;
  return sp;
}

// Kernel shape of a prefill launch: two-tile kernel or not, its tiles mode, and the items.
struct Shape {
  bool pair, tiles;
  int TPC;
  long long items;
};
Shape shape_of(const cp_prefill_args& a, bool fused) {
  Shape sh;
  const int G = a.num_q_heads / a.num_kv_heads;
  // the two-tile kernel unless one head per CTA is forced: two heads of a kv group when they
  // pair up (even G), else two consecutive row tiles of one head (`tiles`)
  sh.pair = a.impl != CP_IMPL_TCGEN05_SINGLE;
  sh.tiles = sh.pair && (G % 2 != 0);
  const int chunk_max = (a.max_seqlen_q + 2 * a.cp - 1) / (2 * a.cp);
  const int span = sh.tiles ? 2 * BM : BM;  // query rows per work item
  sh.TPC = (chunk_max + span - 1) / span;
  sh.items = (long long)2 * a.cp * sh.TPC * a.num_seqs * ((a.kv_shard >= 0 || fused) ? 1 : a.cp) *
             (a.num_q_heads / (sh.pair && !sh.tiles ? 2 : 1));
  return sh;
}

// Pass-KV partials: the item order that keeps the CTAs resident at one time on one kv head of a
// sequence (head groups outermost) when one sequence's K/V is too large for L2 next to the
// outgoing partial rows (>= 64 MB), provided every SM gets many items (>= 32), so that each head
// group's heaviest items starting late does not stretch the grid's tail.  Measured on GB300 at
// 2 x 32768 tokens, cp = 4: 16/16 heads 1339 -> 1554 TFLOP/s, 24/8 +6%, 32/8 +4%, 64/8 +2%;
// at 1 x 8192 (7 items per SM) the same order lost 5-8%, and the fused launch (whose items walk
// a sequence's whole K/V) did not gain.
bool heads_outer_order(const cp_prefill_args& a, const Shape& sh, bool fused, int D) {
  if (a.mode != CP_PASS_KV || fused || a.kv_shard >= 0) return false;
  const double kv_tokens = a.cu_seqlens_kv != nullptr && a.num_seqs > 0
                               ? (double)a.total_kv / a.num_seqs : (double)a.max_seqlen_q;
  if (kv_tokens * a.num_kv_heads * D * 2.0 * 2.0 < 64e6) return false;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  return sh.items >= 32ll * sms;
}

// Split plan of a fused pass-Q launch on the current device (no split for anything else).
SplitPlan fused_split_plan(const cp_prefill_args& a) {
  const Shape sh = shape_of(a, true);
  if (a.mode != CP_PASS_Q || !sh.pair) return SplitPlan{0, 1};
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SplitPlan{0, 1};
  return split_plan(sh.items, a.cp, sms);
}
size_t split_bytes(const SplitPlan& sp, int D) {
  return sp.k > 1 ? (size_t)sp.n_split * sp.k * 2 * BM * (D + 1) * sizeof(float) : 0;
}

template <int D>
cudaError_t launch(const cp_prefill_args& a, float scale, cudaStream_t s, void* fused_out,
                   float* fused_lse, void* ws = nullptr, size_t ws_bytes = 0) {
  CUtensorMap mq, mk, mv;
  const unsigned long long Nq = (unsigned long long)a.total_q;
  if (!make_map(&mq, a.q, (unsigned long long)a.num_q_heads * D, Nq,
                (unsigned long long)a.num_q_heads * D, BM))
    return cudaErrorInvalidValue;
  if (a.mode == CP_PASS_KV) {
    const unsigned long long hd = (unsigned long long)a.num_kv_heads * D;
    const unsigned long long Nkv = a.cu_seqlens_kv ? (unsigned long long)a.total_kv : Nq;
    if (Nkv == 0) return cudaErrorInvalidValue;  // api.cu admits no empty k / v with queries
    if (!make_map(&mk, a.k, hd, Nkv, hd, BN) || !make_map(&mv, a.v, hd, Nkv, hd, BN))
      return cudaErrorInvalidValue;
  }
  const Shape sh = shape_of(a, fused_out != nullptr);
  const bool pair = sh.pair, tiles = sh.tiles;
  int page_kv = 0;
  if (a.mode != CP_PASS_KV) {
    const unsigned long long rows = (unsigned long long)a.cp * a.pool_pages * a.num_kv_heads * 16;
    // pass-Q, two-head kernel, d = 128: one whole-page box per page of K and of V (a quarter
    // of the copies of 64-column x 16-row boxes; the copy engine's per-box cost bounded this
    // path); else 64-column boxes
    if (pair && D == 128 && cp_make_bf16_page_map4(&mk, a.k_cache, rows) &&
        cp_make_bf16_page_map4(&mv, a.v_cache, rows)) {
      page_kv = 1;
    } else if (!make_map(&mk, a.k_cache, D, rows, D, 16) ||
               !make_map(&mv, a.v_cache, D, rows, D, 16)) {
      return cudaErrorInvalidValue;
    }
  }
  TcParams p;
  p.mode = a.mode;
  p.B = a.num_seqs;
  p.Hq = a.num_q_heads;
  p.Hkv = a.num_kv_heads;
  p.cp = a.cp;
  p.I = a.interleave;
  p.max_blocks = a.max_blocks;
  p.q_shard = a.q_shard;
  p.kv_shard = a.kv_shard;
  p.debug = a.debug;
  p.budget = (a.debug & 1) ? (1ll << 21) : kBudget;
  p.TPC = sh.TPC;
  p.f_groups = make_fastdiv((uint32_t)(a.num_q_heads / (pair && !tiles ? 2 : 1)));
  p.f_nslot = make_fastdiv(2u * (uint32_t)a.cp * (uint32_t)(sh.TPC > 0 ? sh.TPC : 1));
  p.f_cp = make_fastdiv((uint32_t)a.cp);
  p.f_tpc = make_fastdiv((uint32_t)(sh.TPC > 0 ? sh.TPC : 1));
  p.f_2cp = make_fastdiv(2u * (uint32_t)a.cp);
  p.f_G = make_fastdiv((uint32_t)(a.num_q_heads / a.num_kv_heads));
  p.Nq = a.total_q;
  p.pool = a.pool_pages;
  p.scale_log2 = scale * kLog2e;
  p.cu_q = a.cu_seqlens_q;
  p.cu_kv = a.mode == CP_PASS_KV ? a.cu_seqlens_kv : nullptr;
  p.seq_lens_kv = a.seq_lens_kv;
  p.tables = a.block_tables;
  p.out = a.out;
  p.lse = a.lse;
  p.err = a.err;
  p.fused = fused_out != nullptr;
  p.out_final = static_cast<__nv_bfloat16*>(fused_out);
  p.lse_final = fused_lse;
  p.heads_outer = heads_outer_order(a, sh, p.fused, D) ? 1 : 0;
  p.row_out = (reinterpret_cast<uintptr_t>(p.fused ? fused_out : static_cast<void*>(a.out)) & 15u) == 0;
  long long grid = sh.items;
  if (grid == 0) return cudaSuccess;
  p.n_whole = (int)(grid < (1ll << 31) ? grid : 0);
  p.split_k = 1;
  p.ws_out = p.ws_lse = nullptr;
  SplitPlan sp{0, 1};
  if (p.fused && a.mode == CP_PASS_Q && pair && ws != nullptr) {
    sp = fused_split_plan(a);
    if (sp.k > 1 && ws_bytes >= split_bytes(sp, D) && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0) {
      p.n_whole = (int)(grid - sp.n_split);
      p.split_k = sp.k;
      p.ws_out = static_cast<float*>(ws);
      p.ws_lse = p.ws_out + (size_t)sp.n_split * sp.k * 2 * BM * D;
      grid = p.n_whole + sp.n_split * sp.k;
    } else {
      sp = SplitPlan{0, 1};
    }
  }
  if (grid >= (1ll << 31)) return cudaErrorInvalidConfiguration;
  cudaError_t e;
  if (pair) {
    const int smem = Layout2<D>::kAlloc;
    // pass-Q at d = 128 (page_kv): K and V pages arrive as whole-page boxes laid out
    // [page][row group][half][8 rows][128 B] in the slot
    // fused pass-Q walks every rank's pages (a variant of its own, so the other kernels keep
    // their registers)
    const bool fq = p.fused && a.mode == CP_PASS_Q;
    auto pick = [&](auto tt) {
      constexpr bool TTv = decltype(tt)::value;
      return fq ? (page_kv ? prefill_tc2_kernel<D, (D == 128), TTv, true>
                           : prefill_tc2_kernel<D, false, TTv, true>)
                : (page_kv ? prefill_tc2_kernel<D, (D == 128), TTv, false>
                           : prefill_tc2_kernel<D, false, TTv, false>);
    };
    auto kern = tiles ? pick(std::true_type{}) : pick(std::false_type{});
    // the warpgroups' register budgets assume the 168 registers a thread of this launch gets; a
    // build that gave the kernel another count would leave an increase waiting, so refuse it
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != 168) return cudaErrorInvalidKernelImage;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, kThreads2, smem, s>>>(mq, mk, mv, p);
    if (sp.k > 1) {
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      // the pieces' partials -> the split items' output rows, scheduled while the attention
      // kernel's last CTAs finish
      cudaLaunchConfig_t cfg;
      std::memset(&cfg, 0, sizeof(cfg));
      cfg.gridDim = dim3((unsigned)sp.n_split);
      cfg.blockDim = dim3(256);
      cfg.stream = s;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      at[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      e = tiles ? cudaLaunchKernelEx(&cfg, fq_split_merge_kernel<D, true>, p)
                : cudaLaunchKernelEx(&cfg, fq_split_merge_kernel<D, false>, p);
      if (e != cudaSuccess) return e;
    }
  } else {
    const int smem = Layout<D>::kAlloc;
    e = cudaFuncSetAttribute(prefill_tc1_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    prefill_tc1_kernel<D><<<(unsigned)grid, kThreads, smem, s>>>(mq, mk, mv, p);
  }
  return cudaGetLastError();
}

}  // namespace
}  // namespace cpattn

bool cp_make_bf16_map_2d(void* map, const void* base, unsigned long long cols,
                         unsigned long long rows, unsigned long long pitch_elems,
                         unsigned box_rows) {
  return cpattn::make_map(static_cast<CUtensorMap*>(map), base, cols, rows, pitch_elems, box_rows);
}

bool cp_make_bf16_page_map4(void* map, const void* base, unsigned long long rows) {
  cpattn::EncodeTiledFn fn = cpattn::encode_fn();
  if (fn == nullptr || rows % 8 != 0) return false;
  cuuint64_t dims[4] = {64, 8, 2, rows / 8};
  cuuint64_t strides[3] = {128 * 2, 128, 8 * 128 * 2};  // next row; second half; next 8 rows
  cuuint32_t box[4] = {64, 8, 2, 2};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool cp_make_bf16_page_map(void* map, const void* base, unsigned long long rows) {
  cpattn::EncodeTiledFn fn = cpattn::encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {64, rows, 2};
  cuuint64_t strides[2] = {128 * 2, 128};  // next row; the second 64-column half
  cuuint32_t box[3] = {64, 16, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool cp_prefill_tc_supported(const cp_prefill_args& a) {
  if (a.dtype != CP_BF16) return false;
  if (a.head_dim != 64 && a.head_dim != 128) return false;
  if (a.mode == CP_PASS_Q && a.block_size != 16) return false;
  return true;
}

cudaError_t cp_launch_prefill_tc(const cp_prefill_args& a, float scale, cudaStream_t s) {
  return a.head_dim == 64 ? cpattn::launch<64>(a, scale, s, nullptr, nullptr)
                          : cpattn::launch<128>(a, scale, s, nullptr, nullptr);
}

cudaError_t cp_launch_prefill_fused(const cp_prefill_args& a, float scale, void* out, float* lse,
                                    void* ws, size_t ws_bytes, cudaStream_t s) {
  return a.head_dim == 64 ? cpattn::launch<64>(a, scale, s, out, lse, ws, ws_bytes)
                          : cpattn::launch<128>(a, scale, s, out, lse, ws, ws_bytes);
}

size_t cp_prefill_fused_split_bytes(const cp_prefill_args& a) {
  return cpattn::split_bytes(cpattn::fused_split_plan(a), a.head_dim);
}
