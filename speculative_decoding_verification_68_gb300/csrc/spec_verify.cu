// spec_verify: batched speculative-decoding verification by rejection sampling
// on one GB300 (sm_103a).  The C interface and the method are described in
// include/spec_verify.h; this file holds the kernels and the host side.
//
// Design (every logit row is streamed from HBM once):
//   * A "unit" is one position of one chain: the pair (target row i, draft
//     row i) for i < k, or the single bonus target row k.  Every unit is
//     processed by one thread-block cluster of C CTAs (C <= 8); CTA r owns the
//     vocabulary slice [r*Vs, (r+1)*Vs) of both rows, and warp w of the CTA a
//     contiguous range of WV 16-byte vectors of that slice.
//   * The kernel is persistent: each cluster walks units cluster_id,
//     cluster_id + n_clusters, ...  Two CTAs share an SM (one, for the
//     largest vocabularies, which need twice the registers).  Each CTA has one
//     shared-memory stage; a bulk (TMA) copy lands the next unit's slice there
//     while the current unit is processed from registers.  The last warp to
//     copy its part out of the stage issues the next copy.
//   * Pass A (registers): per-row maximum, then sum of exp2(z*c - R) with an
//     integer reference R = ceil(max*c), c = log2(e)/T.  Integer references
//     make every rescale between warps and CTAs an exact power of two.
//   * Exchange (DSMEM, no cluster barrier): every warp sends its (max, sum,
//     integer reference) of both rows to every CTA with st.async, which
//     completes the bytes on the receiver's mbarrier; warp 0 of each CTA
//     merges the C*8 parts (in the same order in every CTA, so all CTAs hold
//     identical row statistics) and hands them to the other warps through
//     shared memory and a named barrier.
//   * Pass B (registers): with e_j = 2^(z_j*c - R) and r = S_t/S_d, the
//     residual weight w_j = max(0, e_t - r*e_d) = S_t * max(0, p_j - q_j) (one
//     rounding, exactly zero for identical rows).  Each warp writes the sum of
//     w over its range (and its share of sum e_t) to a small workspace; the
//     CTA owning the drafted token evaluates the accept test.
//   * A finalize kernel (one warp per chain) finds the first rejection tau
//     with a ballot, adds the per-warp masses into the TV distances, locates
//     the warp range holding u * (total mass) of unit tau, re-reads that one
//     range (1/(8C) of the rows) and finishes the inverse-CDF draw.
//   Greedy chains (T == 0) use only the maximum and its lowest index.
//   Units are taken position-major (u = position * B + chain).
//
// Variants of the same kernel (compile-time flags): ENT also sums e*a in pass
// A and writes the entropy of every row; LAZY walks each chain position by
// position and stops at its first rejection (spec_verify_lazy).  A second kernel,
// sv_grad_kernel, uses the same clusters, stage and exchange for the TV and
// overlap losses and their draft-logit gradients (spec_verify_loss_grad).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#include <mutex>

#include "spec_verify.h"

namespace {

constexpr int NT = 256;            // threads per CTA
constexpr int NWARP = NT / 32;
constexpr int CMAX = 8;            // largest cluster
constexpr int ITEMS_MAX = CMAX * NWARP;
constexpr int SMALL_BYTES = 4352;  // bookkeeping area in front of the stage
constexpr float LOG2E_F = 1.44269504088896341f;
constexpr float LN2_F = 0.69314718055994531f;
constexpr float REF_LIMIT = 4194304.0f;   // |max * c| must stay below 2^22
constexpr unsigned FULL = 0xffffffffu;

// status bits of a unit
constexpr int ST_TEMP = 1, ST_TOKEN = 2, ST_ROW = 4;

// Per-unit statistics kept for the finalize kernel.
struct alignas(16) UnitStat {
  float c;       // log2(e) / T, 0 for greedy units
  float R_t;     // integer references of the target / draft row
  float R_d;
  float r;       // S_t / S_d
  float S_t;     // sum_j 2^(z_j c - R_t) over the target row
  int status;    // 0 valid, else ST_* bits
  int greedy;
  int pad;
};

struct KParams {
  const void* target;        // [B, k+1, V]
  const void* draft;         // [B, k, V]
  const int32_t* tokens;     // [B, k]
  const float* temperature;  // [B]
  const float* uniforms;     // [B, k+1]
  float* out_p;              // [B, k] or null
  float* out_q;              // [B, k] or null
  float* out_tv;             // [B, k] or null (greedy units only; others in finalize)
  float* out_ent_t;          // [B, k+1] per-row entropy of the target rows (entropy kernels only)
  float* out_ent_d;          // [B, k]   per-row entropy of the draft rows (entropy kernels only)
  int32_t* ws_acc;           // [B, k]
  int32_t* ws_y;             // [B, k+1] greedy tokens
  UnitStat* ws_stat;         // [B, k+1]
  float* ws_w;               // [B, k+1, items] residual (or target) mass per warp range
  float* ws_p;               // [B, k+1, items] share of sum e_t per warp range
  int* flags;                // [0] invalid count, [1] wait timeout
  int B, k, V, Vs;
  int rbase, rextra;         // rounds of 32 vectors per warp: rbase, one more for the last rextra warps
  int units_per_chain;       // k+1 (verify) or k (TV only)
  int tv_only;
  int tma;                   // bulk copies into the stage
  int vec16;                 // without them: rows 16-byte aligned, so 16-byte loads
  // loss-gradient kernel
  const float* weights;      // [B, k] or null (all 1)
  float* out_loss;           // [B, k] or null
  void* grad;                // [B, k, V] in the logit dtype
  int loss_kind;             // SV_LOSS_TV or SV_LOSS_OVERLAP
  int grad_vec;              // gradient rows can take 16-byte stores
  // lazy verification
  int* ws_grab;              // chains handed out so far past the static ones (zeroed before the launch)
  // verification kernel: tensor-memory columns each CTA allocates (a power of 2; CTAs per SM x this <= 512)
  int tmem_cols;
};

struct alignas(16) X1 {       // one warp's part of the exchange (32 bytes)
  float m_t, m_d;              // maxima of the warp's range in the target / draft row
  float s_t, s_d;              // sums of 2^(z*c - ref) over the range
  int i_t, i_d;                // lowest index of the maximum (T == 0)
  int ref_t, ref_d;            // the integer references ceil(m*c) (NO_REF for an empty range)
};
constexpr int NO_REF = -0x7fffffff - 1;

// Row statistics of one unit, merged by warp 0 of each CTA and read by the others.
struct alignas(16) Merged {
  float S_t, S_d;      // sums of 2^(z*c - R) over the whole rows
  float R_t, R_d;      // integer references of the rows
  float r;             // S_t / S_d
  int IR_t;            // R_t as an integer (NO_REF if the row has no finite maximum)
  int status;          // ST_* bits, 0 if valid
  int cont;            // lazy verification: the chain goes on to the next position
  int grab;            // lazy verification: the counter value rank 0 drew for this unit (-1: none)
  int IR_d;            // a bonus pair: the second row's integer reference (NO_REF as for IR_t)
  int status_d;        // a bonus pair: the second row's ST_* bits
};

struct Small {
  unsigned long long bar;      // stage mbarrier
  unsigned long long xbar[2];  // exchange mbarriers, one per slot set (peers complete their bytes)
  unsigned cnt;                // warps done copying the current stage
  float gz_t, gz_d;            // logits at the drafted token (thread 0 of the owner CTA; lazy: of every CTA)
  float gz_u;                  // lazy verification: the uniform of the accept test
  X1 x1[2][ITEMS_MAX];         // double-buffered exchange slots, written by peers
  int grab[2];                 // lazy verification: rank 0's counter value, per slot set
  Merged mg[2];                // merged row statistics (warp 0 to the other warps), per slot set
  uint32_t tmem;               // the verification instance: this CTA's TMEM columns
};
static_assert(sizeof(Small) <= SMALL_BYTES, "bookkeeping area too small");

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ unsigned cl_rank() { unsigned r; asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r)); return r; }
__device__ __forceinline__ unsigned cl_size() { unsigned r; asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r)); return r; }
__device__ __forceinline__ unsigned cl_id() { unsigned r; asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r)); return r; }
__device__ __forceinline__ unsigned cl_count() { unsigned r; asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r)); return r; }
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint32_t peer_addr(uint32_t a, unsigned rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

// Asynchronous remote store of one exchange part; completes its 32 bytes on
// the receiver's mbarrier (no fence or barrier on the sender's side).
__device__ __forceinline__ void st_async_x1(uint32_t slot, const X1& v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
               ::"r"(slot), "r"(__float_as_uint(v.m_t)), "r"(__float_as_uint(v.m_d)), "r"(__float_as_uint(v.s_t)),
               "r"(__float_as_uint(v.s_d)), "r"(rbar) : "memory");
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
               ::"r"(slot + 16), "r"(v.i_t), "r"(v.i_d), "r"(v.ref_t), "r"(v.ref_d), "r"(rbar) : "memory");
}
__device__ __forceinline__ void st_async_b32(uint32_t slot, int v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(slot), "r"(v), "r"(rbar)
               : "memory");
}
__device__ __forceinline__ void mbar_init(uint32_t a, unsigned n) { asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(n) : "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) { asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory"); }
__device__ __forceinline__ bool mbar_try(uint32_t a, unsigned parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(a), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait for a stage: gives up (and flags the handle) instead of hanging.
// Once any wait has given up, the others see the flag and return within 256 polls.
constexpr int WAIT_POLLS = 1 << 18;   // about 1 s: a poll suspends for ~3.8 us on GB300
// A 4-byte asynchronous copy from global to shared memory, and the wait for
// this thread's copies.
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(saddr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void mbar_wait_bounded(uint32_t a, unsigned parity, int* flags, int polls = WAIT_POLLS) {
  for (int it = 0; it < polls; ++it) {
    if (mbar_try(a, parity)) return;
    if ((it & 255) == 255 && *(volatile int*)&flags[1]) return;
  }
  atomicExch(&flags[1], 1);
}
// Bounded wait for data that peers of the cluster deliver (acquire at cluster scope).
__device__ __forceinline__ void mbar_wait_cluster_bounded(uint32_t a, unsigned parity, int* flags,
                                                          int polls = WAIT_POLLS) {
  for (int it = 0; it < polls; ++it) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(a), "r"(parity) : "memory");
    if (ok) return;
    if ((it & 255) == 255 && *(volatile int*)&flags[1]) return;
  }
  atomicExch(&flags[1], 1);
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, unsigned bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ float ex2(float x) { float y; asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x)); return y; }
__device__ __forceinline__ float nanmax(float a, float b) { float y; asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b)); return y; }
__device__ __forceinline__ float warp_max_nan(float v) { float y; asm volatile("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(y) : "f"(v)); return y; }
__device__ __forceinline__ unsigned warp_min_u32(unsigned v) { unsigned y; asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(y) : "r"(v)); return y; }
typedef unsigned long long u64;
__device__ __forceinline__ u64 pk(float lo, float hi) { u64 r; asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi)); return r; }
__device__ __forceinline__ void upk(u64 v, float& lo, float& hi) { asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v)); }
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) { u64 d; asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c)); return d; }
__device__ __forceinline__ u64 add2(u64 a, u64 b) { u64 d; asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b)); return d; }
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
// Integer log2-domain reference ceil(m*c) of a range maximum m; NO_REF for a range
// without a finite maximum (or beyond the supported range).
__device__ __forceinline__ int iref_of(float m, float c) {
  const float r = ceilf(m * c);
  return (isfinite(m) && fabsf(r) < REF_LIMIT) ? (int)r : NO_REF;
}
// 2^(a - b) for integer references a <= b (exact; 0 below the normal range or for NO_REF)
__device__ __forceinline__ float pow2_diff(int a, int b) {
  const int d = a == NO_REF ? -1000 : a - b;
  return d < -126 ? 0.0f : __int_as_float((d + 127) << 23);
}
__device__ __forceinline__ int warp_max_s32(int v) { int y; asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(y) : "r"(v)); return y; }

// ------------------------------------------------------------ per-type access
// Arrive on the stage counter; the last of NWARP warps returns true (acq_rel,
// so every warp's reads of the stage happen before the caller's next copy).
__device__ __forceinline__ bool stage_release_last(unsigned* cnt) {
  unsigned old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;" : "=r"(old) : "r"(saddr(cnt)) : "memory");
  if (old == NWARP - 1) {
    asm volatile("st.relaxed.cta.shared::cta.u32 [%0], 0;" ::"r"(saddr(cnt)) : "memory");
    return true;
  }
  return false;
}
template <typename Tl> struct Lay;
template <> struct Lay<float> {
  static constexpr int EPV = 4;
  __device__ static uint4 neg_inf() { uint32_t n = 0xff800000u; return make_uint4(n, n, n, n); }
  __device__ static float elem(const uint4& v, int e) {
    uint32_t w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    return __uint_as_float(w);
  }
  __device__ static float load_scalar(const void* p, long long i) { return ((const float*)p)[i]; }
};
template <> struct Lay<__nv_bfloat16> {
  static constexpr int EPV = 8;
  __device__ static uint4 neg_inf() { uint32_t n = 0xff80ff80u; return make_uint4(n, n, n, n); }
  __device__ static float elem(const uint4& v, int e) {
    uint32_t w = (e >> 1) == 0 ? v.x : (e >> 1) == 1 ? v.y : (e >> 1) == 2 ? v.z : v.w;
    return (e & 1) ? bf_hi(w) : bf_lo(w);
  }
  __device__ static float load_scalar(const void* p, long long i) {
    return __uint_as_float((uint32_t)((const uint16_t*)p)[i] << 16);
  }
};

// Unscaled residual weights of one pair of elements: max(0, e_t - r * e_d)
// with e = 2^(z*c - R) and r = S_t / S_d, i.e. S_t * max(0, p - q).  One
// rounding after an exact product, so identical rows give exactly zero.
// The clamp is the fma's saturation to [0, 1], which is exact here: the row
// reference R is at least the row maximum times c, so e_t <= 1 and
// e_t - r * e_d <= 1.  (The packed fma has no saturating form.)
__device__ __forceinline__ float fma_sat(float a, float b, float c) {
  float d;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ u64 pair_w(float t0, float t1, float d0, float d1, u64 cc, u64 nrt, u64 nrd, float nr) {
  float at0, at1, ad0, ad1;
  upk(fma2(pk(t0, t1), cc, nrt), at0, at1);
  upk(fma2(pk(d0, d1), cc, nrd), ad0, ad1);
  return pk(fma_sat(ex2(ad0), nr, ex2(at0)), fma_sat(ex2(ad1), nr, ex2(at1)));
}
// Unscaled target weights of one pair of elements: e_t = S_t * p.
__device__ __forceinline__ u64 pair_p(float t0, float t1, u64 cc, u64 nrt) {
  float at0, at1;
  upk(fma2(pk(t0, t1), cc, nrt), at0, at1);
  return pk(ex2(at0), ex2(at1));
}

// Sum of the weights of one vector (residual if PAIR, else target).
template <typename Tl, bool PAIR>
__device__ __forceinline__ float vec_weight_sum(const uint4& t, const uint4& d, u64 cc, u64 nrt, u64 nrd, float nr) {
  u64 acc;
  if constexpr (sizeof(Tl) == 4) {
    if (PAIR) acc = add2(pair_w(__uint_as_float(t.x), __uint_as_float(t.y), __uint_as_float(d.x), __uint_as_float(d.y), cc, nrt, nrd, nr),
                         pair_w(__uint_as_float(t.z), __uint_as_float(t.w), __uint_as_float(d.z), __uint_as_float(d.w), cc, nrt, nrd, nr));
    else acc = add2(pair_p(__uint_as_float(t.x), __uint_as_float(t.y), cc, nrt), pair_p(__uint_as_float(t.z), __uint_as_float(t.w), cc, nrt));
  } else {
    if (PAIR)
      acc = add2(add2(pair_w(bf_lo(t.x), bf_hi(t.x), bf_lo(d.x), bf_hi(d.x), cc, nrt, nrd, nr),
                      pair_w(bf_lo(t.y), bf_hi(t.y), bf_lo(d.y), bf_hi(d.y), cc, nrt, nrd, nr)),
                 add2(pair_w(bf_lo(t.z), bf_hi(t.z), bf_lo(d.z), bf_hi(d.z), cc, nrt, nrd, nr),
                      pair_w(bf_lo(t.w), bf_hi(t.w), bf_lo(d.w), bf_hi(d.w), cc, nrt, nrd, nr)));
    else
      acc = add2(add2(pair_p(bf_lo(t.x), bf_hi(t.x), cc, nrt), pair_p(bf_lo(t.y), bf_hi(t.y), cc, nrt)),
                 add2(pair_p(bf_lo(t.z), bf_hi(t.z), cc, nrt), pair_p(bf_lo(t.w), bf_hi(t.w), cc, nrt)));
  }
  float lo, hi;
  upk(acc, lo, hi);
  return lo + hi;
}

// Individual weights of one vector (same arithmetic as above, element by element).
template <typename Tl>
__device__ __forceinline__ void vec_weights(const uint4& t, const uint4& d, bool pair, u64 cc, u64 nrt, u64 nrd, float nr,
                                            float (&w)[Lay<Tl>::EPV]) {
  constexpr int EPV = Lay<Tl>::EPV;
#pragma unroll
  for (int e = 0; e < EPV; e += 2) {
    float t0 = Lay<Tl>::elem(t, e), t1 = Lay<Tl>::elem(t, e + 1);
    u64 r;
    if (pair) r = pair_w(t0, t1, Lay<Tl>::elem(d, e), Lay<Tl>::elem(d, e + 1), cc, nrt, nrd, nr);
    else r = pair_p(t0, t1, cc, nrt);
    upk(r, w[e], w[e + 1]);
  }
}

// One 16-byte vector v of a row slice read with plain loads (any alignment);
// entries at or past slen, or when !valid, are -inf.
template <typename Tl>
__device__ __forceinline__ uint4 load_vec_direct(const void* slice, long long v, int slen, bool valid) {
  constexpr int EPV = Lay<Tl>::EPV, ES = (int)sizeof(Tl);
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t x = 0;
#pragma unroll
    for (int h = 0; h < 4 / ES; ++h) {   // 1 fp32 or 2 bf16 per 32-bit word
      const long long idx = v * EPV + q * (4 / ES) + h;
      const bool in = valid && idx < slen;
      if (ES == 4) x = in ? ((const uint32_t*)slice)[idx] : 0xff800000u;
      else x |= (in ? (uint32_t)((const uint16_t*)slice)[idx] : 0xff80u) << (16 * h);
    }
    w[q] = x;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Running maximum over vectors (NaN-propagating).
template <typename Tl> struct MaxAcc;
template <> struct MaxAcc<float> {
  float m = -INFINITY;
  __device__ __forceinline__ void add(const uint4& v) {
    m = nanmax(m, nanmax(nanmax(__uint_as_float(v.x), __uint_as_float(v.y)), nanmax(__uint_as_float(v.z), __uint_as_float(v.w))));
  }
  __device__ __forceinline__ float get() const { return m; }
};
template <> struct MaxAcc<__nv_bfloat16> {
  __nv_bfloat162 m;
  __device__ __forceinline__ MaxAcc() { const uint32_t n = 0xff80ff80u; m = *reinterpret_cast<const __nv_bfloat162*>(&n); }
  __device__ __forceinline__ void add(const uint4& v) {
    m = __hmax2_nan(m, *reinterpret_cast<const __nv_bfloat162*>(&v.x));
    m = __hmax2_nan(m, *reinterpret_cast<const __nv_bfloat162*>(&v.y));
    m = __hmax2_nan(m, *reinterpret_cast<const __nv_bfloat162*>(&v.z));
    m = __hmax2_nan(m, *reinterpret_cast<const __nv_bfloat162*>(&v.w));
  }
  __device__ __forceinline__ float get() const { return nanmax(__low2float(m), __high2float(m)); }
};

// Sum of 2^(z*c + nref) over R vectors with independent packed accumulators
// (the last vector only if `last`: a warp without a last round holds padding there).
template <typename Tl, int R>
__device__ __forceinline__ float rows_expsum(const uint4 (&v)[R], u64 cc, u64 nr, bool last) {
  u64 a0 = 0ull, a1 = 0ull, a2 = 0ull, a3 = 0ull;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    if (j == R - 1 && !last) break;
    float x0, x1, x2, x3;
    if constexpr (sizeof(Tl) == 4) {
      upk(fma2(pk(__uint_as_float(v[j].x), __uint_as_float(v[j].y)), cc, nr), x0, x1);
      upk(fma2(pk(__uint_as_float(v[j].z), __uint_as_float(v[j].w)), cc, nr), x2, x3);
      if (j & 1) { a2 = add2(a2, pk(ex2(x0), ex2(x1))); a3 = add2(a3, pk(ex2(x2), ex2(x3))); }
      else { a0 = add2(a0, pk(ex2(x0), ex2(x1))); a1 = add2(a1, pk(ex2(x2), ex2(x3))); }
    } else {
      float x4, x5, x6, x7;
      upk(fma2(pk(bf_lo(v[j].x), bf_hi(v[j].x)), cc, nr), x0, x1);
      upk(fma2(pk(bf_lo(v[j].y), bf_hi(v[j].y)), cc, nr), x2, x3);
      upk(fma2(pk(bf_lo(v[j].z), bf_hi(v[j].z)), cc, nr), x4, x5);
      upk(fma2(pk(bf_lo(v[j].w), bf_hi(v[j].w)), cc, nr), x6, x7);
      a0 = add2(a0, pk(ex2(x0), ex2(x1)));
      a1 = add2(a1, pk(ex2(x2), ex2(x3)));
      a2 = add2(a2, pk(ex2(x4), ex2(x5)));
      a3 = add2(a3, pk(ex2(x6), ex2(x7)));
    }
  }
  float l0, h0;
  upk(add2(add2(a0, a1), add2(a2, a3)), l0, h0);
  return l0 + h0;
}

// Tensor memory (TMEM, 256 KB per SM: 128 lanes x 512 32-bit columns) holds
// each warp's exponentials from pass A until pass B: lanes 32 * (warp % 4) +
// [0, 32) (the quarter a warp may address), EPV columns per register round,
// warps 4..7 after warps 0..3.  A warp keeps its R target rounds and then the
// draft exponentials of its first DR rounds, DR as many as fit in the CTA's
// share of the columns at the CTAs per SM the kernel is compiled for (two up
// to R = 10, else one).  Stores and loads are asynchronous; the waits below
// order them with the registers that feed or read them.
__host__ __device__ constexpr int tmem_draft_rounds(int epv, int R) {
  return (256 / (R <= 10 ? 2 : 1) - epv * R) / epv < 0 ? 0
       : (256 / (R <= 10 ? 2 : 1) - epv * R) / epv > R ? R
       : (256 / (R <= 10 ? 2 : 1) - epv * R) / epv;   // 256 / CTAs per SM = columns of warps 0..3
}
__host__ __device__ constexpr int tmem_cols_per_warp(int epv, int R) { return epv * (R + tmem_draft_rounds(epv, R)); }
// Only instances whose allocation is 256 or 512 columns use TMEM (R >= 6 in
// bf16, R >= 10 in fp32).  Their CTAs hold at least 86 registers per thread,
// so the register file fits at most two of them on an SM, or one of 512
// columns: whatever mix of this library's kernels shares an SM, its columns
// never exceed 512 and no allocation waits on another of these kernels.  The
// smaller instances (the smallest vocabularies) recompute in pass B instead.
__host__ __device__ constexpr bool tmem_used(int epv, int R) { return 2 * tmem_cols_per_warp(epv, R) > 128; }
template <int EPV, int R>
__device__ __forceinline__ uint32_t tmem_warp_base(uint32_t base) {
  const uint32_t warp = threadIdx.x >> 5;
  return base + ((32u * (warp & 3u)) << 16) + (warp >> 2) * (uint32_t)tmem_cols_per_warp(EPV, R);
}
__device__ __forceinline__ void tmem_st8(uint32_t ta, float e0, float e1, float e2, float e3, float e4, float e5,
                                         float e6, float e7) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               ::"r"(ta), "f"(e0), "f"(e1), "f"(e2), "f"(e3), "f"(e4), "f"(e5), "f"(e6), "f"(e7) : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t ta, float e0, float e1, float e2, float e3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};"
               ::"r"(ta), "f"(e0), "f"(e1), "f"(e2), "f"(e3) : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t ta, float (&e)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(e[0]), "=f"(e[1]), "=f"(e[2]), "=f"(e[3]), "=f"(e[4]), "=f"(e[5]), "=f"(e[6]), "=f"(e[7])
               : "r"(ta) : "memory");
}
__device__ __forceinline__ void tmem_ld4(uint32_t ta, float (&e)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=f"(e[0]), "=f"(e[1]), "=f"(e[2]), "=f"(e[3]) : "r"(ta) : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// rows_expsum, also storing the exponentials of rounds j < NSTORE in this
// warp's TMEM columns (round j at column EPV * j from tm), for pass B to read
// back instead of recomputing.
template <typename Tl, int R, int NSTORE>
__device__ __forceinline__ float rows_expsum_store(const uint4 (&v)[R], u64 cc, u64 nr, bool last, uint32_t tm) {
  u64 a0 = 0ull, a1 = 0ull, a2 = 0ull, a3 = 0ull;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    if (j == R - 1 && !last) break;
    float x0, x1, x2, x3;
    if constexpr (sizeof(Tl) == 4) {
      upk(fma2(pk(__uint_as_float(v[j].x), __uint_as_float(v[j].y)), cc, nr), x0, x1);
      upk(fma2(pk(__uint_as_float(v[j].z), __uint_as_float(v[j].w)), cc, nr), x2, x3);
      const float e0 = ex2(x0), e1 = ex2(x1), e2 = ex2(x2), e3 = ex2(x3);
      if (j < NSTORE) tmem_st4(tm + 4u * j, e0, e1, e2, e3);
      if (j & 1) { a2 = add2(a2, pk(e0, e1)); a3 = add2(a3, pk(e2, e3)); }
      else { a0 = add2(a0, pk(e0, e1)); a1 = add2(a1, pk(e2, e3)); }
    } else {
      float x4, x5, x6, x7;
      upk(fma2(pk(bf_lo(v[j].x), bf_hi(v[j].x)), cc, nr), x0, x1);
      upk(fma2(pk(bf_lo(v[j].y), bf_hi(v[j].y)), cc, nr), x2, x3);
      upk(fma2(pk(bf_lo(v[j].z), bf_hi(v[j].z)), cc, nr), x4, x5);
      upk(fma2(pk(bf_lo(v[j].w), bf_hi(v[j].w)), cc, nr), x6, x7);
      const float e0 = ex2(x0), e1 = ex2(x1), e2 = ex2(x2), e3 = ex2(x3);
      const float e4 = ex2(x4), e5 = ex2(x5), e6 = ex2(x6), e7 = ex2(x7);
      if (j < NSTORE) tmem_st8(tm + 8u * j, e0, e1, e2, e3, e4, e5, e6, e7);
      a0 = add2(a0, pk(e0, e1));
      a1 = add2(a1, pk(e2, e3));
      a2 = add2(a2, pk(e4, e5));
      a3 = add2(a3, pk(e6, e7));
    }
  }
  float l0, h0;
  upk(add2(add2(a0, a1), add2(a2, a3)), l0, h0);
  return l0 + h0;
}

// As rows_expsum, and also sum e*a over the same elements, e = 2^a with
// a = z*c + nref (the log2-domain logit relative to the reference): the
// second moment the row entropy needs, H = ln S - ln2 * (sum e*a) / S.
// a is clamped at -127 so that a masked logit (-inf) adds 0 * -127 instead
// of 0 * -inf; every e is unchanged, since ex2 flushes 2^a to 0 below -126.
__device__ __forceinline__ u64 clamp_m127(u64 x) {
  float lo, hi;
  upk(x, lo, hi);
  return pk(fmaxf(lo, -127.0f), fmaxf(hi, -127.0f));
}
// (The exponentials of rounds j < NSTORE also go to this warp's TMEM columns,
// as in rows_expsum_store.)
template <typename Tl, int R, int NSTORE = 0>
__device__ __forceinline__ float rows_expsum_ent(const uint4 (&v)[R], u64 cc, u64 nr, bool last, float& ea,
                                                 uint32_t tm = 0) {
  u64 a0 = 0ull, a1 = 0ull, a2 = 0ull, a3 = 0ull;
  u64 m0 = 0ull, m1 = 0ull, m2 = 0ull, m3 = 0ull;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    if (j == R - 1 && !last) break;
    u64 x0, x1, x2, x3;
    if constexpr (sizeof(Tl) == 4) {
      x0 = clamp_m127(fma2(pk(__uint_as_float(v[j].x), __uint_as_float(v[j].y)), cc, nr));
      x1 = clamp_m127(fma2(pk(__uint_as_float(v[j].z), __uint_as_float(v[j].w)), cc, nr));
      float p0, p1, p2, p3;
      upk(x0, p0, p1);
      upk(x1, p2, p3);
      const u64 e0 = pk(ex2(p0), ex2(p1)), e1 = pk(ex2(p2), ex2(p3));
      if (j < NSTORE) {
        float f0, f1, f2, f3;
        upk(e0, f0, f1);
        upk(e1, f2, f3);
        tmem_st4(tm + 4u * j, f0, f1, f2, f3);
      }
      if (j & 1) { a2 = add2(a2, e0); a3 = add2(a3, e1); m2 = fma2(e0, x0, m2); m3 = fma2(e1, x1, m3); }
      else { a0 = add2(a0, e0); a1 = add2(a1, e1); m0 = fma2(e0, x0, m0); m1 = fma2(e1, x1, m1); }
    } else {
      x0 = clamp_m127(fma2(pk(bf_lo(v[j].x), bf_hi(v[j].x)), cc, nr));
      x1 = clamp_m127(fma2(pk(bf_lo(v[j].y), bf_hi(v[j].y)), cc, nr));
      x2 = clamp_m127(fma2(pk(bf_lo(v[j].z), bf_hi(v[j].z)), cc, nr));
      x3 = clamp_m127(fma2(pk(bf_lo(v[j].w), bf_hi(v[j].w)), cc, nr));
      float p0, p1, p2, p3, p4, p5, p6, p7;
      upk(x0, p0, p1);
      upk(x1, p2, p3);
      upk(x2, p4, p5);
      upk(x3, p6, p7);
      const u64 e0 = pk(ex2(p0), ex2(p1)), e1 = pk(ex2(p2), ex2(p3)), e2 = pk(ex2(p4), ex2(p5)), e3 = pk(ex2(p6), ex2(p7));
      if (j < NSTORE) {
        float f0, f1, f2, f3, f4, f5, f6, f7;
        upk(e0, f0, f1);
        upk(e1, f2, f3);
        upk(e2, f4, f5);
        upk(e3, f6, f7);
        tmem_st8(tm + 8u * j, f0, f1, f2, f3, f4, f5, f6, f7);
      }
      a0 = add2(a0, e0); a1 = add2(a1, e1); a2 = add2(a2, e2); a3 = add2(a3, e3);
      m0 = fma2(e0, x0, m0); m1 = fma2(e1, x1, m1); m2 = fma2(e2, x2, m2); m3 = fma2(e3, x3, m3);
    }
  }
  float l0, h0, l1, h1;
  upk(add2(add2(m0, m1), add2(m2, m3)), l1, h1);
  ea = l1 + h1;
  upk(add2(add2(a0, a1), add2(a2, a3)), l0, h0);
  return l0 + h0;
}

// Entropy (nats) of a row from its sums relative to the row reference:
// S = sum e, EA = sum e*a with e = 2^a (see rows_expsum_ent).
__device__ __forceinline__ float row_entropy(float S, float EA) { return logf(S) - LN2_F * (EA / S); }

// ------------------------------------------------------------- fused kernel
// A CTA's slice is read in rounds of 32 16-byte vectors (EPV logits each),
// one vector per lane.  Its ceil(nvec / 32) rounds are split over the NWARP
// warps as evenly as possible: every warp takes rbase rounds and the last
// rextra warps one more, so no warp computes a round of padding that a
// lighter split would avoid (at V = 151,552 bf16: 74 rounds, six warps of 9
// and two of 10, instead of eight of 10 with 7.5% padding).  Warp w owns the
// contiguous vectors [warp_vbeg(w), warp_vbeg(w) + 32 * warp_rounds(w)), so
// (rank, warp) items are in vocabulary order; round j, lane l holds vector
// warp_vbeg(w) + 32 j + l.  In shared memory each warp's range of each row has
// its own block of R*32 vectors (R >= every warp's rounds); the tail past
// the range stays -inf, so the copy into registers needs no bounds checks.
__host__ __device__ __forceinline__ int warp_rounds(int w, int rbase, int rextra) {
  return rbase + (w >= NWARP - rextra ? 1 : 0);
}
__host__ __device__ __forceinline__ int warp_vbeg(int w, int rbase, int rextra) {
  const int lo = NWARP - rextra;   // warps with rbase rounds
  return 32 * (w * rbase + (w > lo ? w - lo : 0));
}
// The warp whose range holds vector lv of the slice.
__device__ __forceinline__ int warp_of_vec(int lv, int rbase, int rextra) {
  const int ri = lv >> 5, lo = NWARP - rextra;
  if (ri < lo * rbase) return ri / rbase;
  return lo + (ri - lo * rbase) / (rbase + 1);
}
struct Geo {
  const KParams* p;
  __device__ __forceinline__ unsigned C() const { return cl_size(); }
  __device__ __forceinline__ unsigned rank() const { return cl_rank(); }
  __device__ __forceinline__ int items() const { return (int)cl_size() * NWARP; }
  __device__ __forceinline__ int slice0() const { return (int)cl_rank() * p->Vs; }
  __device__ __forceinline__ int slen() const { return max(0, min(p->Vs, p->V - slice0())); }
  __device__ __forceinline__ int vbeg() const { return warp_vbeg((int)(threadIdx.x >> 5), p->rbase, p->rextra); }
  __device__ __forceinline__ int rounds() const { return warp_rounds((int)(threadIdx.x >> 5), p->rbase, p->rextra); }
};

// Units are taken position-major, u = ipos * B + b for the k verified
// positions, so that every cluster's walk u = cluster_id, cluster_id +
// n_clusters, ... meets every position equally often.  The bonus rows follow.
// With PAIRED (instances of two CTAs per SM) they go two chains to a unit
// (chains b = 2j and b + 1; the last one alone when B is odd): a bonus row
// needs only its row statistics, so a pair of them fills the stage as a row
// pair does and takes one exchange and one merge instead of two.  The pair's
// second row is read after the first (the registers hold one row), so the
// stage is released later; at one CTA per SM nothing hides the next unit's
// copy behind that, and those instances take the bonus rows one at a time.
struct Unit {
  int b, ipos;
};
template <bool PAIRED>
__device__ __forceinline__ Unit unit_of(unsigned u, unsigned B, unsigned k) {
  Unit r;
  if (u < B * k) {
    const unsigned ipos = u / B;
    r.b = (int)(u - ipos * B);
    r.ipos = (int)ipos;
  } else {
    r.b = (int)((PAIRED ? 2u : 1u) * (u - B * k));
    r.ipos = (int)k;
  }
  return r;
}
// Instances whose verification walk pairs the bonus rows.
template <int R> __host__ __device__ constexpr bool pairs_bonus_rows() { return R <= 10; }
// The same for a walk over the k verified positions alone.
__device__ __forceinline__ Unit pos_unit_of(unsigned u, unsigned B) {
  const unsigned ipos = u / B;
  Unit r;
  r.b = (int)(u - ipos * B);
  r.ipos = (int)ipos;
  return r;
}

template <typename Tl> __device__ __forceinline__ int nvec_of(const Geo& g) { return (g.slen() + Lay<Tl>::EPV - 1) / Lay<Tl>::EPV; }

// Lowest global index in this warp's range of a row that holds the warp's
// maximum m (greedy rows).
template <typename Tl, int R>
__device__ __forceinline__ int warp_argmax(const uint4 (&r)[R], float m, const Geo& g) {
  constexpr int EPV = Lay<Tl>::EPV;
  const int lane = threadIdx.x & 31;
  int ci = 0x7fffffff;
#pragma unroll
  for (int j = R - 1; j >= 0; --j) {
#pragma unroll
    for (int e = EPV - 1; e >= 0; --e) {
      const int gi = (int)g.slice0() + (g.vbeg() + j * 32 + lane) * EPV + e;
      if (Lay<Tl>::elem(r[j], e) == m) ci = gi;
    }
  }
  return (int)warp_min_u32((unsigned)ci);
}

// Bulk copies of one unit into the warp blocks of the stage, issued by one
// whole warp: lane 0 arms the mbarrier with the byte count, then lane w
// copies warp w's range of the target row and lane 8 + w that of the draft row.
// With BONUS_PAIRS (the verification walk), a bonus unit of chain b < B - 1
// copies the bonus row of chain b + 1 in place of the draft row.
template <typename Tl, int R, bool BONUS_PAIRS = false>
__device__ __forceinline__ void issue_unit_load(const KParams& P, const Geo& g, Unit n, uint32_t bar,
                                                const unsigned char* stage) {
  constexpr int ES = (int)sizeof(Tl);
  const int lane = threadIdx.x & 31;
  const int k = P.k;
  const bool pair = n.ipos < k;
  const bool two = pair || (BONUS_PAIRS && n.b + 1 < P.B);   // two rows in the stage
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // earlier generic accesses of the stage first
  const long long trow = (long long)n.b * (k + 1) + n.ipos;
  const long long drow = BONUS_PAIRS && !pair ? (long long)(n.b + 1) * (k + 1) + k : (long long)n.b * k + n.ipos;
  if (lane == 0) {
    const unsigned bytes = (unsigned)nvec_of<Tl>(g) * 16u;
    if (bytes > 0) mbar_expect_tx(bar, two ? 2 * bytes : bytes);
    else mbar_arrive(bar);
  }
  __syncwarp();
  const int w = lane & 7, row = lane >> 3;
  if (lane < 16 && (row == 0 || two)) {
    const int vb = warp_vbeg(w, P.rbase, P.rextra);
    const int len = max(0, min(32 * warp_rounds(w, P.rbase, P.rextra), nvec_of<Tl>(g) - vb));
    if (len > 0) {
      const char* src = (const char*)(row == 0 || (BONUS_PAIRS && !pair) ? P.target : P.draft) +
                        ((size_t)(row == 0 ? trow : drow) * P.V + g.slice0()) * ES + (size_t)vb * 16;
      const uint32_t dst = saddr(stage + ((size_t)(row * NWARP + w) * R * 32) * 16);
      bulk_g2s(dst, src, (unsigned)len * 16u, bar);
    }
  }
}

// Named barrier 1 over the whole CTA: warp 0 publishes the merged statistics.
__device__ __forceinline__ void merged_arrive() { asm volatile("bar.arrive 1, %0;" ::"n"(NT) : "memory"); }
__device__ __forceinline__ void merged_wait() { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); }

// A warp's residual mass of its range whose lane sum is still to be taken: the
// five shuffle steps run during the next unit's copy, where they overlap the
// shared-memory loads, instead of at the end of pass B.
struct PendingMass {
  float w;        // this lane's part
  size_t item;    // the range's slot in ws_w
  bool on;
};
__device__ __forceinline__ void flush_mass(const KParams& P, PendingMass* pm) {
  if (pm && pm->on) {
    const float w = warp_sum_f32(pm->w);
    if ((threadIdx.x & 31) == 0) P.ws_w[pm->item] = w;
    pm->on = false;
  }
}

// Unit kinds: a verified position (the target and draft rows of one chain),
// one bonus row, or the bonus rows of two chains (the second one, of chain
// un.b + 1 at temperature T2, in the draft slots).
enum { U_BONUS = 0, U_PAIR = 1, U_BONUS2 = 2 };

// Returns, for lazy verification, whether the chain goes on to its next
// position (the same in every CTA of the cluster); 0 otherwise.
template <typename Tl, int R, int KIND, bool ENT, bool LAZY>
__device__ __forceinline__ int process_unit(const KParams& P, Small& S, const uint4* blk_t, const uint4* blk_d,
                                             const Geo& g, const Unit un, unsigned phase, int& n1, const uint32_t bar,
                                             const unsigned char* smem_stage, const Unit next, bool tma_next,
                                             const float T, const int x, const bool carry = false,
                                             const uint32_t tm = 0, PendingMass* pm = nullptr, const float T2 = 0.0f) {
  constexpr bool PAIR = KIND == U_PAIR;     // a verified position
  constexpr bool B2 = KIND == U_BONUS2;     // two bonus rows
  static_assert(!(B2 && LAZY), "the lazy walk takes bonus rows one at a time");
  constexpr int EPV = Lay<Tl>::EPV;
  constexpr int ES = (int)sizeof(Tl);
  constexpr bool TM = tmem_used(EPV, R);   // exponentials kept in TMEM between the passes
  constexpr int NS_T = TM ? R : 0, NS_D = TM ? tmem_draft_rounds(EPV, R) : 0;   // rounds kept per row
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = P.k, V = P.V;
  const int b = un.b, ipos = un.ipos;

  // Lazy verification takes the accept decision in every CTA at the merge:
  // the logits at the drafted token and the uniform are loaded ahead of it.
  float lz_t = 0.0f, lz_d = 0.0f, lz_u = 0.0f;
  if (LAZY && PAIR && tid == 0 && x >= 0 && x < V) {
    lz_t = Lay<Tl>::load_scalar(P.target, ((long long)b * (k + 1) + ipos) * V + x);
    lz_d = Lay<Tl>::load_scalar(P.draft, ((long long)b * k + ipos) * V + x);
    lz_u = P.uniforms[(size_t)b * (k + 1) + ipos];
  }
  // A unit that carries a grab: rank 0 draws the next counter value now and
  // sends it to every CTA with this unit's exchange.
  int grab_v = 0;
  if (LAZY && carry && tid == 0 && g.rank() == 0) grab_v = atomicAdd(P.ws_grab, 1);

  // ---------------- this warp's vectors of the unit into registers
  uint4 rt[R], rd[R];
  bool own_x = false;
  const bool last = g.rounds() == R;   // warp-uniform: this warp owns a last round
  // This warp is done with the stage; the last warp to finish issues the next unit's copy.
  auto release_stage = [&]() {
    __syncwarp();
    bool fin = false;
    if (lane == 0) fin = stage_release_last(&S.cnt);
    fin = __shfl_sync(FULL, fin, 0);
    if (fin && tma_next) issue_unit_load<Tl, R, !LAZY && pairs_bonus_rows<R>()>(P, g, next, bar, smem_stage);
  };
  if (P.tma) {
    mbar_wait_bounded(bar, phase, P.flags);
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const bool in = j < R - 1 || last;   // else padding: -inf without a load
      rt[j] = in ? blk_t[j * 32 + lane] : Lay<Tl>::neg_inf();
      if (PAIR) rd[j] = in ? blk_d[j * 32 + lane] : Lay<Tl>::neg_inf();
    }
    own_x = !LAZY && PAIR && !P.tv_only && x >= 0 && x < V && (long long)x >= g.slice0() && (long long)x < g.slice0() + g.slen();
    if (PAIR && tid == 0 && own_x) {
      const int lx = (int)(x - g.slice0());
      const int lv = lx / EPV, wb = warp_of_vec(lv, P.rbase, P.rextra), iv = lv - warp_vbeg(wb, P.rbase, P.rextra);
      const unsigned char* bt = smem_stage + ((size_t)(0 * NWARP + wb) * R * 32 + iv) * 16;
      const unsigned char* bd = smem_stage + ((size_t)(1 * NWARP + wb) * R * 32 + iv) * 16;
      S.gz_t = Lay<Tl>::load_scalar(bt, lx % EPV);
      S.gz_d = Lay<Tl>::load_scalar(bd, lx % EPV);
      cp_async4(&S.gz_u, P.uniforms + (size_t)b * (k + 1) + ipos);   // for the accept test, which ends the unit
    }
    flush_mass(P, pm);   // the previous unit's residual mass, while the loads land
    if (!B2) release_stage();   // a bonus pair still needs its second row from the stage
  } else {
    const long long trow = (long long)b * (k + 1) + ipos, drow = (long long)b * k + ipos;
    const char* tb = (const char*)P.target + ((size_t)trow * V + g.slice0()) * ES;
    const char* db = (const char*)P.draft + ((size_t)drow * V + g.slice0()) * ES;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int v = g.vbeg() + j * 32 + lane;
      const bool in = j < g.rounds() && v < nvec_of<Tl>(g);
      if (P.vec16) {   // the tail vector of a 16-byte-aligned row is whole (the row length is too)
        rt[j] = in ? __ldg(reinterpret_cast<const uint4*>(tb) + v) : Lay<Tl>::neg_inf();
        if (PAIR) rd[j] = in ? __ldg(reinterpret_cast<const uint4*>(db) + v) : Lay<Tl>::neg_inf();
      } else {
        rt[j] = load_vec_direct<Tl>(tb, v, g.slen(), in);
        if (PAIR) rd[j] = load_vec_direct<Tl>(db, v, g.slen(), in);
      }
    }
    own_x = !LAZY && PAIR && !P.tv_only && x >= 0 && x < V && (long long)x >= g.slice0() && (long long)x < g.slice0() + g.slen();
    if (PAIR && tid == 0 && own_x) {
      S.gz_t = Lay<Tl>::load_scalar(P.target, trow * V + x);
      S.gz_d = Lay<Tl>::load_scalar(P.draft, drow * V + x);
      cp_async4(&S.gz_u, P.uniforms + (size_t)b * (k + 1) + ipos);
    }
    flush_mass(P, pm);
  }

  if (LAZY && PAIR && tid == 0) {   // parked in shared memory, out of the registers pass A needs
    S.gz_t = lz_t;
    S.gz_d = lz_d;
    S.gz_u = lz_u;
  }

  const bool t_ok = T >= 0.0f && T <= 3.0e38f;   // false for NaN and inf
  const bool greedy = !(T > 0.0f) || !t_ok;      // invalid temperatures take the cheap path
  const bool x_ok = !PAIR || P.tv_only || (x >= 0 && x < V);
  const float c = greedy ? 0.0f : fminf(__fdiv_rn(LOG2E_F, T), 3.0e38f);
  // a bonus pair: the second chain's temperature, taken the same way
  const bool t_ok2 = T2 >= 0.0f && T2 <= 3.0e38f;
  const bool greedy2 = !(T2 > 0.0f) || !t_ok2;
  const float c2 = greedy2 ? 0.0f : fminf(__fdiv_rn(LOG2E_F, T2), 3.0e38f);

  // ---------------- pass A: per-warp statistics, pushed to every CTA of the cluster
  MaxAcc<Tl> mx_t, mx_d;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    if (j == R - 1 && !last) break;
    mx_t.add(rt[j]);
    if (PAIR) mx_d.add(rd[j]);
  }
  X1 mine;
  mine.m_t = warp_max_nan(mx_t.get());
  mine.m_d = PAIR ? warp_max_nan(mx_d.get()) : -INFINITY;
  mine.i_t = 0x7fffffff; mine.i_d = 0x7fffffff;
  mine.s_t = 0.0f; mine.s_d = 0.0f;
  mine.ref_t = NO_REF; mine.ref_d = NO_REF;
  if constexpr (B2) {
    // Each row as a lone bonus row would take it, with its chain's temperature;
    // the second row comes into the registers once the first is done with them.
    float s_t = 0.0f, s_d = 0.0f, ea_t = 0.0f, ea_d = 0.0f;
    if (greedy) {
      mine.i_t = warp_argmax<Tl, R>(rt, mine.m_t, g);
    } else {
      mine.ref_t = iref_of(mine.m_t, c);
      const float rw = mine.ref_t == NO_REF ? 0.0f : (float)mine.ref_t;
      if constexpr (ENT) s_t = rows_expsum_ent<Tl, R>(rt, pk(c, c), pk(-rw, -rw), last, ea_t);
      else mine.s_t = warp_sum_f32(rows_expsum<Tl, R>(rt, pk(c, c), pk(-rw, -rw), last));
    }
    if (P.tma) {
#pragma unroll
      for (int j = 0; j < R; ++j) rd[j] = j < R - 1 || last ? blk_d[j * 32 + lane] : Lay<Tl>::neg_inf();
      release_stage();
    } else {
      const char* db = (const char*)P.target + ((size_t)((long long)(b + 1) * (k + 1) + ipos) * V + g.slice0()) * ES;
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int v = g.vbeg() + j * 32 + lane;
        const bool in = j < g.rounds() && v < nvec_of<Tl>(g);
        rd[j] = P.vec16 ? (in ? __ldg(reinterpret_cast<const uint4*>(db) + v) : Lay<Tl>::neg_inf())
                        : load_vec_direct<Tl>(db, v, g.slen(), in);
      }
    }
    {
      MaxAcc<Tl> mx2;
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (j == R - 1 && !last) break;
        mx2.add(rd[j]);
      }
      mine.m_d = warp_max_nan(mx2.get());
    }
    if (greedy2) {
      mine.i_d = warp_argmax<Tl, R>(rd, mine.m_d, g);
    } else {
      mine.ref_d = iref_of(mine.m_d, c2);
      const float rw = mine.ref_d == NO_REF ? 0.0f : (float)mine.ref_d;
      if constexpr (ENT) s_d = rows_expsum_ent<Tl, R>(rd, pk(c2, c2), pk(-rw, -rw), last, ea_d);
      else mine.s_d = warp_sum_f32(rows_expsum<Tl, R>(rd, pk(c2, c2), pk(-rw, -rw), last));
    }
    if constexpr (ENT) {   // the index fields carry sum e*a for sampling rows
      if (!greedy || !greedy2) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float y0 = __shfl_xor_sync(FULL, s_t, o), y1 = __shfl_xor_sync(FULL, s_d, o);
          const float y2 = __shfl_xor_sync(FULL, ea_t, o), y3 = __shfl_xor_sync(FULL, ea_d, o);
          upk(add2(pk(s_t, s_d), pk(y0, y1)), s_t, s_d);
          upk(add2(pk(ea_t, ea_d), pk(y2, y3)), ea_t, ea_d);
        }
      }
      if (!greedy) { mine.s_t = s_t; mine.i_t = __float_as_int(ea_t); }
      if (!greedy2) { mine.s_d = s_d; mine.i_d = __float_as_int(ea_d); }
    }
  } else if (greedy) {
    int ci_t = 0x7fffffff, ci_d = 0x7fffffff;   // lowest global index holding the warp maximum
#pragma unroll
    for (int j = R - 1; j >= 0; --j) {
#pragma unroll
      for (int e = EPV - 1; e >= 0; --e) {
        const int gi = (int)g.slice0() + (g.vbeg() + j * 32 + lane) * EPV + e;
        if (Lay<Tl>::elem(rt[j], e) == mine.m_t) ci_t = gi;
        if (PAIR && Lay<Tl>::elem(rd[j], e) == mine.m_d) ci_d = gi;
      }
    }
    mine.i_t = (int)warp_min_u32((unsigned)ci_t);
    if (PAIR) mine.i_d = (int)warp_min_u32((unsigned)ci_d);
  } else {
    const u64 cc = pk(c, c);
    mine.ref_t = iref_of(mine.m_t, c);
    const float rwt = mine.ref_t == NO_REF ? 0.0f : (float)mine.ref_t;
    if constexpr (ENT) {   // the index fields carry sum e*a for sampling units
      float ea_t = 0.0f, ea_d = 0.0f;
      if (PAIR) mine.s_t = rows_expsum_ent<Tl, R, NS_T>(rt, cc, pk(-rwt, -rwt), last, ea_t, tm);
      else mine.s_t = rows_expsum_ent<Tl, R>(rt, cc, pk(-rwt, -rwt), last, ea_t);
      if (PAIR) {
        mine.ref_d = iref_of(mine.m_d, c);
        const float rwd = mine.ref_d == NO_REF ? 0.0f : (float)mine.ref_d;
        mine.s_d = rows_expsum_ent<Tl, R, NS_D>(rd, cc, pk(-rwd, -rwd), last, ea_d, tm + EPV * R);
      }
      float v0 = mine.s_t, v1 = mine.s_d, v2 = ea_t, v3 = ea_d;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float y0 = __shfl_xor_sync(FULL, v0, o), y1 = __shfl_xor_sync(FULL, v1, o);
        const float y2 = __shfl_xor_sync(FULL, v2, o), y3 = __shfl_xor_sync(FULL, v3, o);
        upk(add2(pk(v0, v1), pk(y0, y1)), v0, v1);
        upk(add2(pk(v2, v3), pk(y2, y3)), v2, v3);
      }
      mine.s_t = v0; mine.s_d = v1;
      mine.i_t = __float_as_int(v2); mine.i_d = __float_as_int(v3);
    } else {
      // a row pair keeps its target exponentials, and the draft ones of the first
      // rounds, in TMEM for pass B (in the instances that use TMEM)
      mine.s_t = warp_sum_f32(PAIR ? rows_expsum_store<Tl, R, NS_T>(rt, cc, pk(-rwt, -rwt), last, tm)
                                   : rows_expsum<Tl, R>(rt, cc, pk(-rwt, -rwt), last));
      if (PAIR) {
        mine.ref_d = iref_of(mine.m_d, c);
        const float rwd = mine.ref_d == NO_REF ? 0.0f : (float)mine.ref_d;
        mine.s_d = warp_sum_f32(rows_expsum_store<Tl, R, NS_D>(rd, cc, pk(-rwd, -rwd), last, tm + EPV * R));
      }
    }
  }
  const int set1 = n1 & 1;
  const uint32_t xbar = saddr(&S.xbar[set1]);
  if (tid == 0) mbar_expect_tx(xbar, (unsigned)g.items() * 32u + (LAZY && carry ? 4u : 0u));
  if (lane < (int)g.C())
    st_async_x1(peer_addr(saddr(&S.x1[set1][g.rank() * NWARP + warp]), lane), mine, peer_addr(xbar, lane));
  if (LAZY && carry && warp == 0 && g.rank() == 0) {   // cluster-uniform condition
    const int gv = __shfl_sync(FULL, grab_v, 0);
    if (lane < (int)g.C()) st_async_b32(peer_addr(saddr(&S.grab[set1]), lane), gv, peer_addr(xbar, lane));
  }
  const unsigned xpar = (unsigned)((n1 >> 1) & 1);
  ++n1;

  const size_t ui = (size_t)b * (k + 1) + ipos;   // unit index within [B, k+1]
  const size_t pi = (size_t)b * k + ipos;         // position index within [B, k]
  Merged& mg = S.mg[set1];
  if (warp == 0) {
    // Cluster merge (warp 0 only): lane l holds items l and l + 32.
    mbar_wait_cluster_bounded(xbar, xpar, P.flags);
    X1 ia, ib;
    {
      X1 z;
      z.m_t = -INFINITY; z.m_d = -INFINITY; z.s_t = 0.0f; z.s_d = 0.0f; z.i_t = 0x7fffffff; z.i_d = 0x7fffffff;
      z.ref_t = NO_REF; z.ref_d = NO_REF;
      ia = lane < g.items() ? S.x1[set1][lane] : z;
      ib = lane + 32 < g.items() ? S.x1[set1][lane + 32] : z;
    }
    float M_t, M_d;
    int A_t = 0, A_d = 0, IR_t = NO_REF, IR_d = NO_REF;
    float S_t = 0.0f, S_d = 0.0f;
    if constexpr (B2) {   // two independent rows, each merged as a lone bonus row is
      if (greedy) {
        M_t = warp_max_nan(nanmax(ia.m_t, ib.m_t));
        A_t = (int)warp_min_u32((unsigned)min(ia.m_t == M_t ? ia.i_t : 0x7fffffff, ib.m_t == M_t ? ib.i_t : 0x7fffffff));
      } else {
        IR_t = warp_max_s32(max(ia.ref_t, ib.ref_t));
        S_t = warp_sum_f32(ia.s_t * pow2_diff(ia.ref_t, IR_t) + ib.s_t * pow2_diff(ib.ref_t, IR_t));
        M_t = warp_max_nan(nanmax(ia.m_t, ib.m_t));
      }
      if (greedy2) {
        M_d = warp_max_nan(nanmax(ia.m_d, ib.m_d));
        A_d = (int)warp_min_u32((unsigned)min(ia.m_d == M_d ? ia.i_d : 0x7fffffff, ib.m_d == M_d ? ib.i_d : 0x7fffffff));
      } else {
        IR_d = warp_max_s32(max(ia.ref_d, ib.ref_d));
        S_d = warp_sum_f32(ia.s_d * pow2_diff(ia.ref_d, IR_d) + ib.s_d * pow2_diff(ib.ref_d, IR_d));
        M_d = warp_max_nan(nanmax(ia.m_d, ib.m_d));
      }
    } else if (greedy) {
      M_t = warp_max_nan(nanmax(ia.m_t, ib.m_t));
      M_d = PAIR ? warp_max_nan(nanmax(ia.m_d, ib.m_d)) : 0.0f;
      A_t = (int)warp_min_u32((unsigned)min(ia.m_t == M_t ? ia.i_t : 0x7fffffff, ib.m_t == M_t ? ib.i_t : 0x7fffffff));
      if (PAIR)
        A_d = (int)warp_min_u32((unsigned)min(ia.m_d == M_d ? ia.i_d : 0x7fffffff, ib.m_d == M_d ? ib.i_d : 0x7fffffff));
    } else {
      // the row reference is the largest item reference (ceil is monotonic);
      // the maxima, needed only for the status, are reduced after the sums
      IR_t = warp_max_s32(max(ia.ref_t, ib.ref_t));
      if (PAIR) {
        IR_d = warp_max_s32(max(ia.ref_d, ib.ref_d));
        const u64 st = add2(pk(ia.s_t * pow2_diff(ia.ref_t, IR_t), ia.s_d * pow2_diff(ia.ref_d, IR_d)),
                            pk(ib.s_t * pow2_diff(ib.ref_t, IR_t), ib.s_d * pow2_diff(ib.ref_d, IR_d)));
        upk(st, S_t, S_d);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float a = __shfl_xor_sync(FULL, S_t, o), bb = __shfl_xor_sync(FULL, S_d, o);
          upk(add2(pk(S_t, S_d), pk(a, bb)), S_t, S_d);
        }
      } else {
        S_t = warp_sum_f32(ia.s_t * pow2_diff(ia.ref_t, IR_t) + ib.s_t * pow2_diff(ib.ref_t, IR_t));
      }
      M_t = warp_max_nan(nanmax(ia.m_t, ib.m_t));
      M_d = PAIR ? warp_max_nan(nanmax(ia.m_d, ib.m_d)) : 0.0f;
    }
    const float R_t = IR_t == NO_REF ? 0.0f : (float)IR_t, R_d = IR_d == NO_REF ? 0.0f : (float)IR_d;
    bool row_ok = isfinite(M_t) && (!PAIR || isfinite(M_d));
    if (!greedy) {
      row_ok = row_ok && fabsf(M_t * c) < REF_LIMIT && S_t > 0.0f && isfinite(S_t);
      if (PAIR) row_ok = row_ok && fabsf(M_d * c) < REF_LIMIT && S_d > 0.0f && isfinite(S_d);
    }
    const int status = (t_ok ? 0 : ST_TEMP) | (x_ok ? 0 : ST_TOKEN) | (row_ok ? 0 : ST_ROW);
    int status_d = 0;   // a bonus pair: the second row's status, taken the same way
    if constexpr (B2) {
      bool ok2 = isfinite(M_d);
      if (!greedy2) ok2 = ok2 && fabsf(M_d * c2) < REF_LIMIT && S_d > 0.0f && isfinite(S_d);
      status_d = (t_ok2 ? 0 : ST_TEMP) | (ok2 ? 0 : ST_ROW);
    }
    // q_j = e_d * r / S_t, correctly rounded: equal sums give r = 1 exactly, so
    // identical rows keep an exactly zero residual.
    const float r_f = PAIR && !greedy ? S_t / S_d : 0.0f;
    Merged m;
    if (lane == 0) {
      int cont = 0;   // the same test as the accept test below, on the same values
      if (LAZY && PAIR && status == 0) {
        if (greedy) {
          cont = x == A_t;
        } else {
          const float lpx = fmaf(S.gz_t, c, -R_t), lqx = fmaf(S.gz_d, c, -R_d);
          cont = S.gz_u < exp2f(lpx - lqx) * (S_d / S_t);
        }
      }
      m.S_t = S_t; m.S_d = S_d; m.R_t = R_t; m.R_d = R_d; m.r = r_f; m.IR_t = IR_t; m.status = status; m.cont = cont;
      m.grab = LAZY && carry ? S.grab[set1] : -1;
      m.IR_d = IR_d; m.status_d = status_d;
      mg = m;
    }
    __syncwarp();
    merged_arrive();
    if (ENT && g.rank() == 0) {
      // Row entropies, by rank 0 alone (the only CTA that writes them) and
      // after the other warps are released.  Each item's sum e*a is relative
      // to its own reference; on the row reference it becomes
      // 2^(ref_i - R) * (EA_i + (ref_i - R) * s_i).
      float H_t = __int_as_float(0x7fc00000), H_d = H_t;
      auto part = [&](float s_i, float ea_i, int ref_i, int IR) {   // empty ranges and padding add 0
        return ref_i == NO_REF ? 0.0f : pow2_diff(ref_i, IR) * fmaf((float)ref_i - (float)IR, s_i, ea_i);
      };
      if constexpr (B2) {   // each row with its own temperature
        if (greedy && t_ok && isfinite(M_t)) H_t = 0.0f;
        if (greedy2 && t_ok2 && isfinite(M_d)) H_d = 0.0f;
        if (!greedy || !greedy2) {
          float e_t = part(ia.s_t, __int_as_float(ia.i_t), ia.ref_t, IR_t) + part(ib.s_t, __int_as_float(ib.i_t), ib.ref_t, IR_t);
          float e_d = part(ia.s_d, __int_as_float(ia.i_d), ia.ref_d, IR_d) + part(ib.s_d, __int_as_float(ib.i_d), ib.ref_d, IR_d);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float y0 = __shfl_xor_sync(FULL, e_t, o), y1 = __shfl_xor_sync(FULL, e_d, o);
            upk(add2(pk(e_t, e_d), pk(y0, y1)), e_t, e_d);
          }
          const bool ok_t = t_ok && isfinite(M_t) && fabsf(M_t * c) < REF_LIMIT && S_t > 0.0f && isfinite(S_t);
          const bool ok_d = t_ok2 && isfinite(M_d) && fabsf(M_d * c2) < REF_LIMIT && S_d > 0.0f && isfinite(S_d);
          if (!greedy && ok_t) H_t = row_entropy(S_t, e_t);
          if (!greedy2 && ok_d) H_d = row_entropy(S_d, e_d);
        }
      } else if (greedy) {   // the one-hot greedy distribution (NaN for an invalid temperature)
        if (t_ok && isfinite(M_t)) H_t = 0.0f;
        if (t_ok && PAIR && isfinite(M_d)) H_d = 0.0f;
      } else {
        float e_t = part(ia.s_t, __int_as_float(ia.i_t), ia.ref_t, IR_t) + part(ib.s_t, __int_as_float(ib.i_t), ib.ref_t, IR_t);
        float e_d = PAIR ? part(ia.s_d, __int_as_float(ia.i_d), ia.ref_d, IR_d) + part(ib.s_d, __int_as_float(ib.i_d), ib.ref_d, IR_d)
                         : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float y0 = __shfl_xor_sync(FULL, e_t, o), y1 = __shfl_xor_sync(FULL, e_d, o);
          upk(add2(pk(e_t, e_d), pk(y0, y1)), e_t, e_d);
        }
        const bool ok_t = t_ok && isfinite(M_t) && fabsf(M_t * c) < REF_LIMIT && S_t > 0.0f && isfinite(S_t);
        const bool ok_d = t_ok && isfinite(M_d) && fabsf(M_d * c) < REF_LIMIT && S_d > 0.0f && isfinite(S_d);
        if (ok_t) H_t = row_entropy(S_t, e_t);
        if (PAIR && ok_d) H_d = row_entropy(S_d, e_d);
      }
      if (lane == 0) {
        P.out_ent_t[ui] = H_t;
        if (PAIR) P.out_ent_d[pi] = H_d;
        if (B2) P.out_ent_t[(size_t)(b + 1) * (k + 1) + ipos] = H_d;
      }
    }
    // rank 0's workspace writes come after the other warps are released: only
    // the finalize kernel reads them
    if (lane == 0) {
      if (g.rank() == 0) {
        UnitStat st;
        st.c = c; st.R_t = R_t; st.R_d = B2 ? 0.0f : R_d; st.r = r_f; st.S_t = S_t;
        st.status = status; st.greedy = greedy ? 1 : 0; st.pad = 0;
        P.ws_stat[ui] = st;
        if constexpr (B2) {   // the second chain's bonus row, as its own unit would write it
          const size_t ui2 = (size_t)(b + 1) * (k + 1) + ipos;
          UnitStat s2;
          s2.c = c2; s2.R_t = R_d; s2.R_d = 0.0f; s2.r = 0.0f; s2.S_t = S_d;
          s2.status = status_d; s2.greedy = greedy2 ? 1 : 0; s2.pad = 0;
          P.ws_stat[ui2] = s2;
          if (greedy2 && status_d == 0) P.ws_y[ui2] = A_d;
        }
        if (status != 0 || greedy) {
          if (!P.tv_only && status == 0) {
            P.ws_y[ui] = A_t;
            if (PAIR) {
              P.ws_acc[pi] = x == A_t;
              if (P.out_p) P.out_p[pi] = x == A_t ? 1.0f : 0.0f;
              if (P.out_q) P.out_q[pi] = x == A_d ? 1.0f : 0.0f;
            }
          }
          if (LAZY && PAIR && status != 0) P.ws_acc[pi] = 0;   // an invalid position stops the chain
          if (PAIR && status != 0) {   // no probabilities at an invalid position
            if (P.out_p) P.out_p[pi] = __int_as_float(0x7fc00000);
            if (P.out_q) P.out_q[pi] = __int_as_float(0x7fc00000);
          }
          if (PAIR && P.out_tv) P.out_tv[pi] = status == 0 ? (A_t != A_d ? 1.0f : 0.0f) : __int_as_float(0x7fc00000);
        } else if (LAZY && PAIR) {
          P.ws_acc[pi] = m.cont;
        }
      }
    }
  } else {
    merged_wait();
  }
  const Merged M = mg;
  if constexpr (B2) {   // each sampling row's per-range target mass, as for a lone bonus row
    const int it = (int)g.rank() * NWARP + warp;
    if (M.status == 0 && !greedy) {
      const float pmass = mine.s_t * pow2_diff(mine.ref_t, M.IR_t);
      if (lane == 0) { P.ws_p[ui * ITEMS_MAX + it] = pmass; P.ws_w[ui * ITEMS_MAX + it] = pmass; }
    }
    if (M.status_d == 0 && !greedy2) {
      const size_t ui2 = (size_t)(b + 1) * (k + 1) + ipos;
      const float pmass = mine.s_d * pow2_diff(mine.ref_d, M.IR_d);
      if (lane == 0) { P.ws_p[ui2 * ITEMS_MAX + it] = pmass; P.ws_w[ui2 * ITEMS_MAX + it] = pmass; }
    }
    return 0;
  }
  // cluster-uniform; an accepted position of a lazy walk needs no residual
  if (M.status != 0 || greedy || (LAZY && M.cont)) {
    if (!LAZY && own_x && tid == 0) cp_async_wait_all();   // no accept test: the copied uniform is not used
    return M.cont;
  }

  // this range's part of S_t (the target mass, and the draw from p when the residual is zero)
  const float pmass = mine.s_t * pow2_diff(mine.ref_t, M.IR_t);
  const size_t item = ui * ITEMS_MAX + g.rank() * NWARP + warp;
  if (!PAIR) {   // the bonus row: its mass is already known
    if (lane == 0) { P.ws_p[item] = pmass; P.ws_w[item] = pmass; }
    return 0;
  }
  if (lane == 0) P.ws_p[item] = pmass;

  // ---------------- pass B: residual mass of this warp's range
  const u64 cc = pk(c, c);
  float wacc = 0.0f;
  {
    // The target exponentials e_t = 2^(z_t c - ref_t) come back from TMEM
    // (pass A stored them, relative to this warp's reference ref_t), as do the
    // draft ones of the first rounds; the rest are recomputed relative to the
    // warp's references, as in pass A (all of them in the instances without
    // TMEM).  With s_t = 2^(ref_t - R_t) and s_d = 2^(ref_d - R_d) (exact
    // powers of 2), the weight on the row references is
    //   max(0, s_t e_t - r s_d e_d) = s_t * sat(e_t - r (s_d / s_t) e_d),
    // the clamp being exact because e_t <= 1; identical rows give exactly 0.
    if (mine.ref_t != NO_REF) {   // else the warp's target range is all masked: no residual
      constexpr int EPV = Lay<Tl>::EPV;
      const int e_sc = mine.ref_d == NO_REF ? 0 : (mine.ref_d - (int)M.R_d) - (mine.ref_t - M.IR_t);
      const float sc = e_sc < -126 ? 0.0f : e_sc > 127 ? INFINITY : __int_as_float((e_sc + 127) << 23);
      const float nrs = mine.ref_d == NO_REF ? 0.0f : -M.r * sc;
      const float rwd = mine.ref_d == NO_REF ? 0.0f : (float)mine.ref_d;
      const u64 nrdw = pk(-rwd, -rwd);
      const float rwt = (float)mine.ref_t;
      const u64 nrtw = pk(-rwt, -rwt);
      if (TM) tmem_wait_st();   // pass A's stores are complete
      constexpr int ndr = NS_D;   // rounds whose draft exponentials were kept too
      const uint32_t tmd = tm + EPV * R;
      u64 a0 = 0ull, a1 = 0ull;
      // one round: the weights of its EPV positions, from e_t and e_d (kept, or recomputed as in pass A)
      auto round_w = [&](int j, const float (&et)[EPV], const float (&ed)[EPV], bool kept) {
#pragma unroll
        for (int q = 0; q < EPV / 2; ++q) {
          float e0, e1;
          if (kept) {
            e0 = ed[2 * q];
            e1 = ed[2 * q + 1];
          } else {
            float ad0, ad1;
            if constexpr (EPV == 8) {
              const uint32_t wd = q == 0 ? rd[j].x : q == 1 ? rd[j].y : q == 2 ? rd[j].z : rd[j].w;
              upk(fma2(pk(bf_lo(wd), bf_hi(wd)), cc, nrdw), ad0, ad1);
            } else {
              const uint32_t wd0 = q == 0 ? rd[j].x : rd[j].z, wd1 = q == 0 ? rd[j].y : rd[j].w;
              upk(fma2(pk(__uint_as_float(wd0), __uint_as_float(wd1)), cc, nrdw), ad0, ad1);
            }
            e0 = ex2(ad0);
            e1 = ex2(ad1);
          }
          const u64 w = pk(fma_sat(e0, nrs, et[2 * q]), fma_sat(e1, nrs, et[2 * q + 1]));
          if (q & 1) a1 = add2(a1, w); else a0 = add2(a0, w);
        }
      };
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (j == R - 1 && !last) break;
        const bool kept = j < ndr;
        float et[EPV], ed[EPV];
        if constexpr (!TM) {   // recomputed as in pass A
#pragma unroll
          for (int q = 0; q < EPV / 2; ++q) {
            float a0t, a1t;
            if constexpr (EPV == 8) {
              const uint32_t wt = q == 0 ? rt[j].x : q == 1 ? rt[j].y : q == 2 ? rt[j].z : rt[j].w;
              upk(fma2(pk(bf_lo(wt), bf_hi(wt)), cc, nrtw), a0t, a1t);
            } else {
              const uint32_t wt0 = q == 0 ? rt[j].x : rt[j].z, wt1 = q == 0 ? rt[j].y : rt[j].w;
              upk(fma2(pk(__uint_as_float(wt0), __uint_as_float(wt1)), cc, nrtw), a0t, a1t);
            }
            et[2 * q] = ex2(a0t);
            et[2 * q + 1] = ex2(a1t);
          }
        } else if constexpr (EPV == 8) {
          tmem_ld8(tm + 8u * j, et);
          if (kept) tmem_ld8(tmd + 8u * j, ed);
        } else {
          tmem_ld4(tm + 4u * j, et);
          if (kept) tmem_ld4(tmd + 4u * j, ed);
        }
        if (TM) tmem_wait_ld();
        round_w(j, et, ed, kept);
      }
      float l, h;
      upk(add2(a0, a1), l, h);
      wacc = (l + h) * pow2_diff(mine.ref_t, M.IR_t);
    }
  }
  if (pm) {   // summed over the lanes during the next unit's copy (or after the last unit)
    pm->w = wacc;
    pm->item = item;
    pm->on = true;
  } else {
    const float wwarp = warp_sum_f32(wacc);
    if (lane == 0) P.ws_w[item] = wwarp;
  }
  if (!LAZY && own_x && tid == 0) {   // accept test at the drafted token
    const float lpx = fmaf(S.gz_t, c, -M.R_t), lqx = fmaf(S.gz_d, c, -M.R_d);
    const float ratio = exp2f(lpx - lqx) * (M.S_d / M.S_t);
    cp_async_wait_all();   // the uniform copied in at the start of the unit
    const float u_acc = S.gz_u;
    P.ws_acc[pi] = u_acc < ratio ? 1 : 0;
    if (P.out_p) P.out_p[pi] = exp2f(lpx) / M.S_t;
    if (P.out_q) P.out_q[pi] = exp2f(lqx) / M.S_d;
  }
  return 0;
}

template <typename Tl, int R, bool ENT, bool LAZY>
__global__ void __launch_bounds__(NT, R <= 10 ? 2 : 1) sv_fused_kernel(const KParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  Small& S = *reinterpret_cast<Small*>(smem);
  unsigned char* stage = smem + SMALL_BYTES;   // [2 rows][NWARP][R*32] vectors

  const int tid = threadIdx.x, warp = tid >> 5;
  Geo g;
  g.p = &P;
  const unsigned cid = cl_id(), ncl = cl_count();
  const int k = P.k;
  const unsigned B = (unsigned)P.B;
  // the verified positions, then the bonus rows (verification only), paired where the instance pairs them
  constexpr bool PB = pairs_bonus_rows<R>();
  const unsigned n_units = B * (unsigned)k + (P.units_per_chain > k ? (PB ? (B + 1u) >> 1 : B) : 0u);   // below 2^31
  const uint32_t bar = saddr(&S.bar);
  const uint4* blk_t = reinterpret_cast<const uint4*>(stage) + (size_t)(0 * NWARP + warp) * R * 32;
  const uint4* blk_d = reinterpret_cast<const uint4*>(stage) + (size_t)(1 * NWARP + warp) * R * 32;

  if (P.tma) {   // the tails of the warp blocks stay -inf for the whole kernel
    uint4* st = reinterpret_cast<uint4*>(stage);
    for (int i = tid; i < 2 * NWARP * R * 32; i += NT) st[i] = Lay<Tl>::neg_inf();
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(saddr(&S.xbar[0]), 1);
    mbar_init(saddr(&S.xbar[1]), 1);
    S.cnt = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  constexpr bool USE_TMEM = tmem_used(Lay<Tl>::EPV, R);   // exponentials wait in TMEM from pass A to pass B
  if (USE_TMEM && warp == 0) {   // the host keeps CTAs per SM x tmem_cols within the SM's 512 columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&S.tmem)),
                 "r"(P.tmem_cols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (USE_TMEM) asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (USE_TMEM) asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  cluster_sync_all();   // every peer's shared memory is live before the first remote store
  const uint32_t tm = USE_TMEM ? tmem_warp_base<Lay<Tl>::EPV, R>(S.tmem) : 0u;

  unsigned phase = 0;
  int n1 = 0;   // exchanges performed (selects the slot set)
  if constexpr (LAZY) {
    // Each cluster walks chains position by position and stops a chain at its
    // first rejection (or after its bonus row).  Two chains are in flight,
    // taking turns, so that the unit after the current one is always known
    // (the other chain's next position, decided one unit earlier) and its
    // copy can be issued ahead.  A third chain waits in reserve.
    // Chains are handed out at run time: each cluster starts with chains
    // cluster_id + j * n_clusters, j < 3; when the reserve is taken, the next
    // unit's exchange carries a value of a global counter that rank 0 bumps,
    // and chain 3 * n_clusters + value becomes the reserve.  The walk is the
    // same in every CTA of the cluster: it depends only on the accept
    // decisions, which every CTA takes from the merged statistics, and on the
    // counter values, which every CTA receives.
    const unsigned first = 3u * ncl;
    auto chain_or_none = [&](unsigned long long c) { return c < B ? (int)c : -1; };
    Unit cur, nxt;
    cur.b = chain_or_none(cid); cur.ipos = 0;
    nxt.b = chain_or_none(cid + (unsigned long long)ncl); nxt.ipos = 0;
    int reserve = chain_or_none(cid + 2ull * ncl);
    bool refill = false;      // the reserve was taken: the next unit carries a grab
    bool exhausted = cid + 2ull * ncl >= B;
    bool loaded = false;      // cur's copy was issued while the previous unit ran
    while (cur.b >= 0) {
      if (P.tma && !loaded) {   // nothing issued ahead: every warp is done with the stage
        __syncthreads();
        if (warp == 0) issue_unit_load<Tl, R>(P, g, cur, bar, stage);
      }
      const bool has_next = nxt.b >= 0;
      const float T = P.temperature[cur.b];
      const int x = cur.ipos < k ? P.tokens[(size_t)cur.b * k + cur.ipos] : 0;
      const bool carry = refill;
      int cont;
      if (cur.ipos < k)
        cont = process_unit<Tl, R, U_PAIR, ENT, true>(P, S, blk_t, blk_d, g, cur, phase, n1, bar, stage, nxt,
                                                     P.tma && has_next, T, x, carry, tm);
      else
        cont = process_unit<Tl, R, U_BONUS, ENT, true>(P, S, blk_t, blk_d, g, cur, phase, n1, bar, stage, nxt,
                                                      P.tma && has_next, T, x, carry, tm);
      phase ^= 1u;
      if (carry) {   // this unit's exchange brought the new reserve
        reserve = chain_or_none(first + (unsigned long long)(unsigned)S.mg[(n1 - 1) & 1].grab);
        exhausted = reserve < 0;
        refill = false;
      }
      Unit after;
      if (cont) {
        after.b = cur.b; after.ipos = cur.ipos + 1;
      } else {
        after.b = reserve; after.ipos = 0;
        if (reserve >= 0) { reserve = -1; refill = !exhausted; }
      }
      if (has_next) { cur = nxt; nxt = after; loaded = true; }
      else { cur = after; loaded = false; }
    }
  } else {
    unsigned u = cid;
    Unit cur = unit_of<PB>(u, B, (unsigned)k);
    if (P.tma && warp == 0 && u < n_units) issue_unit_load<Tl, R, PB>(P, g, cur, bar, stage);
    PendingMass pm;
    pm.on = false;
    for (; u < n_units; u += ncl, phase ^= 1u) {
      const bool has_next = u + ncl < n_units;
      const Unit next = unit_of<PB>(u + ncl, B, (unsigned)k);
      const float T = P.temperature[cur.b];
      const int x = cur.ipos < k && !P.tv_only ? P.tokens[(size_t)cur.b * k + cur.ipos] : 0;
      const bool tma_next = P.tma && has_next;
      if (cur.ipos < k)
        process_unit<Tl, R, U_PAIR, ENT, false>(P, S, blk_t, blk_d, g, cur, phase, n1, bar, stage, next, tma_next, T,
                                                x, false, tm, &pm);
      else if (PB && cur.b + 1 < (int)B)
        process_unit<Tl, R, U_BONUS2, ENT, false>(P, S, blk_t, blk_d, g, cur, phase, n1, bar, stage, next, tma_next,
                                                  T, 0, false, tm, &pm, P.temperature[cur.b + 1]);
      else
        process_unit<Tl, R, U_BONUS, ENT, false>(P, S, blk_t, blk_d, g, cur, phase, n1, bar, stage, next, tma_next, T,
                                                 x, false, tm, &pm);
      cur = next;
    }
    flush_mass(P, &pm);
  }
  if (USE_TMEM) {   // every TMEM access of the CTA is complete before its columns are freed
    tmem_wait_st();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(S.tmem), "r"(P.tmem_cols) : "memory");
    }
  }
  cluster_sync_all();   // no CTA leaves while a peer could still address its shared memory
}

// Self-test of the bounded waits: thread 0 waits on an mbarrier that nothing
// completes, with the stage wait and then with the cluster-scope wait; both
// must give up.  No copy or remote store is in flight, so nothing is left
// pending when the CTA exits.
__global__ void sv_wait_selftest_kernel(int* flags, int polls, long long* cycles) {
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x == 0) {
    mbar_init(saddr(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const long long t0 = clock64();
    mbar_wait_bounded(saddr(&bar), 0u, flags, polls);
    const long long t1 = clock64();
    mbar_wait_cluster_bounded(saddr(&bar), 0u, flags, polls);   // the flag is set: returns early
    const long long t2 = clock64();
    cycles[0] = t1 - t0;
    cycles[1] = t2 - t1;
  }
}

// ------------------------------------------------------------ finalize kernel
struct FParams {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const float* uniforms;
  const int32_t* ws_acc;
  const int32_t* ws_y;
  const UnitStat* ws_stat;
  const float* ws_w;
  const float* ws_p;
  int32_t* out_tokens;
  int32_t* out_tau;
  float* out_tv;
  int* flags;
  int B, k, V, Vs, rbase, rextra, items, vec16, tv_only;   // vec16: rows 16-byte aligned
  int lazy;   // positions after the first rejection were not verified
};

// One warp per chain: tau by ballot, TV from the per-range masses, and the
// inverse-CDF draw of the final token (re-reading only the owning range).
template <typename Tl, int R>
__global__ void __launch_bounds__(256) sv_finalize_kernel(const FParams F) {
  constexpr int EPV = Lay<Tl>::EPV;
  constexpr int ES = (int)sizeof(Tl);
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (b >= F.B) return;
  const int k = F.k, items = F.items;
  const size_t ub = (size_t)b * (k + 1);
  const int npos = F.tv_only ? k : k + 1;
  // Everything that does not depend on tau is loaded first, together: the
  // accept bits (not written, and not used, for TV only), the statistics and
  // greedy token of every unit (lane i holds position i's), the drafted
  // tokens and the uniform of the final draw.
  const int a = lane < k ? F.ws_acc[(size_t)b * k + lane] : 1;
  UnitStat sl;
  sl.c = 0.0f; sl.R_t = 0.0f; sl.R_d = 0.0f; sl.r = 0.0f; sl.S_t = 1.0f; sl.status = 0; sl.greedy = 0; sl.pad = 0;
  int yl = 0;
  if (lane < npos) {
    sl = F.ws_stat[ub + lane];
    yl = F.ws_y[ub + lane];
  }
  const int tok = !F.tv_only && lane < k ? F.tokens[(size_t)b * k + lane] : -1;
  const float u_fin = F.tv_only ? 0.0f : F.uniforms[ub + k];   // the final draw uses u[b, k]
  // A bounded wait that gave up (in this call, or in an earlier one whose flag
  // has not been cleared by spec_verify_get_error) leaves the statistics
  // unreliable: every chain is then reported invalid, and every TV is NaN.
  const bool timed_out = *(volatile const int*)&F.flags[1] != 0;

  const unsigned rej = __ballot_sync(FULL, lane < k && a == 0);
  const int tau = rej ? __ffs(rej) - 1 : k;
  // the last position whose unit was verified: a lazy walk stopped at the first rejection
  const int last = F.lazy ? tau : npos - 1;
  const bool bad = __any_sync(FULL, lane <= last && sl.status != 0);

  // TV of every valid, non-greedy position: 8 positions per pass, 4 lanes per
  // position, each lane adding 16 consecutive range masses (loaded together)
  if (F.out_tv) {
    for (int i0 = 0; i0 < k; i0 += 8) {
      const int i = i0 + (lane >> 2), q = lane & 3;
      const int src = min(i, k - 1);   // every lane takes part in the shuffles
      const int st_i = __shfl_sync(FULL, sl.status, src), gr_i = __shfl_sync(FULL, sl.greedy, src);
      const float S_t = __shfl_sync(FULL, sl.S_t, src);
      const bool ok = i < k && st_i == 0 && !gr_i;
      float v = 0.0f;
      if (i < k) {
        const float4* w4 = reinterpret_cast<const float4*>(F.ws_w + (ub + i) * ITEMS_MAX) + q * 4;
        float4 w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = w4[e];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int it = q * 16 + e * 4;   // ranges past `items` were never written
          v += (it < items ? w[e].x : 0.0f) + (it + 1 < items ? w[e].y : 0.0f) +
               (it + 2 < items ? w[e].z : 0.0f) + (it + 3 < items ? w[e].w : 0.0f);
        }
      }
      v += __shfl_xor_sync(FULL, v, 1);
      v += __shfl_xor_sync(FULL, v, 2);
      if (q == 0 && ok) F.out_tv[(size_t)b * k + i] = v / S_t;
    }
    if (timed_out && lane < k) F.out_tv[(size_t)b * k + lane] = __int_as_float(0x7fc00000);
  }
  if (bad && !timed_out && lane == 0) atomicAdd(&F.flags[0], 1);
  if (F.tv_only) return;
  if (bad || timed_out) {
    if (lane <= k) F.out_tokens[ub + lane] = -1;
    if (lane == 0) F.out_tau[b] = -1;
    return;
  }
  const bool pair = tau < k;
  const size_t uu = ub + tau;
  UnitStat us;   // unit tau's statistics, from lane tau
  us.c = __shfl_sync(FULL, sl.c, tau); us.R_t = __shfl_sync(FULL, sl.R_t, tau);
  us.R_d = __shfl_sync(FULL, sl.R_d, tau); us.r = __shfl_sync(FULL, sl.r, tau);
  us.S_t = __shfl_sync(FULL, sl.S_t, tau); us.status = 0; us.pad = 0;
  us.greedy = __shfl_sync(FULL, sl.greedy, tau);
  const int y_greedy = __shfl_sync(FULL, yl, tau);
  int y = 0;
  if (us.greedy) {
    y = y_greedy;
  } else {
    // ---- which (CTA, warp) range holds u * total mass
    const float* wp = F.ws_w + uu * ITEMS_MAX;
    const float* pp = F.ws_p + uu * ITEMS_MAX;
    const int ka = 2 * lane, kb = 2 * lane + 1;
    float fa = ka < items ? wp[ka] : 0.0f, fb = kb < items ? wp[kb] : 0.0f;
    const bool fallback = pair && !(warp_sum_f32(fa + fb) > 0.0f);   // zero residual: draw from p
    if (fallback) {
      fa = ka < items ? pp[ka] : 0.0f;
      fb = kb < items ? pp[kb] : 0.0f;
    }
    const double wa = fa, wb = fb;
    double incl = wa + wb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += t;
    }
    double excl = __shfl_up_sync(FULL, incl, 1);
    if (lane == 0) excl = 0.0;
    const double total = __shfl_sync(FULL, incl, 31);
    const double tt = (double)u_fin * total;
    const bool ca = wa > 0.0 && tt < excl + wa;
    const bool cb = wb > 0.0 && tt < incl;
    const unsigned hit = __ballot_sync(FULL, ca || cb);
    int item;
    bool over;
    double tloc;
    if (hit) {
      const int L = __ffs(hit) - 1;
      const bool la = __shfl_sync(FULL, ca, L);
      item = 2 * L + (la ? 0 : 1);
      tloc = tt - __shfl_sync(FULL, la ? excl : excl + wa, L);
      over = false;
    } else {
      const unsigned pos = __ballot_sync(FULL, wa > 0.0 || wb > 0.0);
      const int L = pos ? 31 - __clz(pos) : 0;
      item = 2 * L + (__shfl_sync(FULL, wb > 0.0, L) ? 1 : 0);
      tloc = 0.0;
      over = true;
    }
    // ---- re-read the owning range and finish the draw there
    const int crank = item / NWARP, cwarp = item % NWARP;
    const long long slice0 = (long long)crank * F.Vs;
    const int slen = (int)max(0LL, min((long long)F.Vs, (long long)F.V - slice0));
    const int nvec = (slen + EPV - 1) / EPV;
    const int vbeg = warp_vbeg(cwarp, F.rbase, F.rextra);
    const int vend = min(vbeg + 32 * warp_rounds(cwarp, F.rbase, F.rextra), nvec);
    const bool use_pair = pair && !fallback;
    const char* tb = (const char*)F.target + ((size_t)(ub + tau) * F.V + slice0) * ES;
    const char* db = (const char*)F.draft + (((size_t)b * k + (pair ? tau : 0)) * F.V + slice0) * ES;
    uint4 rt[R], rd[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int v = vbeg + j * 32 + lane;
      if (F.vec16) {
        rt[j] = v < vend ? __ldg(reinterpret_cast<const uint4*>(tb) + v) : Lay<Tl>::neg_inf();
        rd[j] = (use_pair && v < vend) ? __ldg(reinterpret_cast<const uint4*>(db) + v) : Lay<Tl>::neg_inf();
      } else {
        rt[j] = load_vec_direct<Tl>(tb, v, slen, v < vend);
        rd[j] = load_vec_direct<Tl>(db, v, slen, use_pair && v < vend);
      }
    }
    const u64 cc = pk(us.c, us.c);
    const u64 nrt = pk(-us.R_t, -us.R_t), nrd = pk(-us.R_d, -us.R_d);
    const float nr = -us.r;
    float wl[R];
#pragma unroll
    for (int j = 0; j < R; ++j)
      wl[j] = use_pair ? vec_weight_sum<Tl, true>(rt[j], rd[j], cc, nrt, nrd, nr)
                       : vec_weight_sum<Tl, false>(rt[j], rd[j], cc, nrt, nrd, nr);
    int jstar = -1, jlast = -1;
    double tin = 0.0, run = 0.0;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const double tj = (double)warp_sum_f32(wl[j]);
      if (tj > 0.0) jlast = j;
      if (!over && jstar < 0 && tj > 0.0 && tloc < run + tj) { jstar = j; tin = tloc - run; }
      run += tj;
    }
    if (jstar < 0) { jstar = jlast; over = true; }
    if (jstar < 0) jstar = 0;   // no positive weight in the range (cannot happen for a valid unit)
    float mw = 0.0f;
#pragma unroll
    for (int j = 0; j < R; ++j) if (j == jstar) mw = wl[j];
    double inc = (double)mw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(FULL, inc, o);
      if (lane >= o) inc += t;
    }
    const unsigned h2 = __ballot_sync(FULL, !over && mw > 0.0f && tin < inc);
    const unsigned p2 = __ballot_sync(FULL, mw > 0.0f);
    int lstar;
    if (h2) lstar = __ffs(h2) - 1;
    else { lstar = p2 ? 31 - __clz(p2) : 0; over = true; }
    const double t2 = tin - (__shfl_sync(FULL, inc, lstar) - (double)__shfl_sync(FULL, mw, lstar));
    int estar = -1;
    if (lane == lstar) {
      float w[EPV];
#pragma unroll
      for (int e = 0; e < EPV; ++e) w[e] = 0.0f;
#pragma unroll
      for (int j = 0; j < R; ++j)
        if (j == jstar) vec_weights<Tl>(rt[j], rd[j], use_pair, cc, nrt, nrd, nr, w);
      int elast = 0;
      double run2 = 0.0;
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        if (w[e] > 0.0f) elast = e;
        if (!over && estar < 0 && w[e] > 0.0f && t2 < run2 + (double)w[e]) estar = e;
        run2 += (double)w[e];
      }
      if (estar < 0) estar = elast;
    }
    estar = __shfl_sync(FULL, estar, lstar);
    y = (int)slice0 + (vbeg + jstar * 32 + lstar) * EPV + estar;
  }
  if (lane <= k) F.out_tokens[ub + lane] = lane < tau ? tok : lane == tau ? y : -1;
  if (lane == 0) F.out_tau[b] = tau;
}

// ------------------------------------------------------- loss-gradient kernel
// Per position i of chain b (target row i, draft row i), from the two rows
// held in registers:
//   pass A and the first exchange: row statistics, as in the fused kernel;
//   pass B: e_t = 2^(z_t c - R_t), e_d = 2^(z_d c - R_d), the indicator
//     [q < p] = [e_t - r e_d > 0] (one bit per element, kept for pass C), and
//     per warp B1 = sum_{q<p} e_d, B2 = sum_{q>=p} e_t;
//   second exchange: beta = B1 / S_d, alpha = (r B1 + B2) / S_t = sum min(p, q);
//   pass C: d(w l)/d z_d = K e_d ([q < p] - beta), K = w dl/dalpha / (T S_d),
//     written in the logit dtype.
// Loss: TV = 1 - alpha (SV_LOSS_TV) or -ln alpha (SV_LOSS_OVERLAP).

__device__ __forceinline__ u64 mul2(u64 a, u64 b) { u64 d; asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b)); return d; }
// Two fp32 values as one bf16x2 word (lo in the low half), rounded to nearest even.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// One 16-byte vector of gradients, already in the logit dtype (EPV values
// packed in w), into the draft-gradient row `row` at slice-relative vector v;
// entries at or past slen are not written.
template <typename Tl>
__device__ __forceinline__ void store_grad(void* row, int v, int slen, bool vec_ok, const uint4& w) {
  constexpr int EPV = Lay<Tl>::EPV, ES = (int)sizeof(Tl);
  const int e0 = v * EPV;
  if (e0 >= slen) return;
  if (vec_ok && e0 + EPV <= slen) {
    reinterpret_cast<uint4*>(row)[v] = w;
    return;
  }
#pragma unroll
  for (int e = 0; e < EPV; ++e) {
    if (e0 + e >= slen) break;
    const uint32_t word = (e * ES) / 4 == 0 ? w.x : (e * ES) / 4 == 1 ? w.y : (e * ES) / 4 == 2 ? w.z : w.w;
    if constexpr (ES == 4) reinterpret_cast<uint32_t*>(row)[e0 + e] = word;
    else reinterpret_cast<uint16_t*>(row)[e0 + e] = (uint16_t)((e & 1) ? (word >> 16) : (word & 0xffffu));
  }
}

// Sum of 32-byte exchange items l and l + 32 over the warp, for the s_t and s_d fields.
__device__ __forceinline__ void warp_sum_items(const X1* it, int items, float& a, float& d) {
  const int lane = threadIdx.x & 31;
  float a0 = lane < items ? it[lane].s_t : 0.0f, d0 = lane < items ? it[lane].s_d : 0.0f;
  float a1 = lane + 32 < items ? it[lane + 32].s_t : 0.0f, d1 = lane + 32 < items ? it[lane + 32].s_d : 0.0f;
  u64 v = add2(pk(a0, d0), pk(a1, d1));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float x, y;
    upk(v, x, y);
    v = add2(v, pk(__shfl_xor_sync(FULL, x, o), __shfl_xor_sync(FULL, y, o)));
  }
  upk(v, a, d);
}

// A scheduling fence between vectors: the next vector's registers are made to
// depend on the accumulator, so the compiler keeps one vector in flight per
// thread instead of hoisting every exponential of the unrolled loop (which
// spills at 128 registers).
__device__ __forceinline__ void fence_vec(uint4& a, uint4& b, u64& acc) {
  asm volatile("" : "+r"(a.x), "+r"(a.y), "+r"(a.z), "+r"(a.w), "+r"(b.x), "+r"(b.y), "+r"(b.z), "+r"(b.w), "+l"(acc));
}

struct alignas(16) GradStat {   // the second merge, published by warp 0
  float beta, K;
  int ok, pad;
};

template <typename Tl, int R>
__device__ __forceinline__ void grad_unit(const KParams& P, Small& S, GradStat* gs, const uint4* blk_t,
                                          const uint4* blk_d, const Geo& g, const Unit un, unsigned phase, int& n1,
                                          const uint32_t bar, const unsigned char* smem_stage, const Unit next,
                                          bool tma_next, const float T) {
  constexpr int EPV = Lay<Tl>::EPV;
  constexpr int ES = (int)sizeof(Tl);
  constexpr int NBW = (R * EPV + 31) / 32;   // indicator words per thread
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = P.k, V = P.V;
  const int b = un.b, ipos = un.ipos;
  const long long trow = (long long)b * (k + 1) + ipos, drow = (long long)b * k + ipos;

  uint4 rt[R], rd[R];
  const bool last = g.rounds() == R;   // warp-uniform: this warp owns a last round
  if (P.tma) {
    mbar_wait_bounded(bar, phase, P.flags);
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const bool in = j < R - 1 || last;   // else padding: -inf without a load
      rt[j] = in ? blk_t[j * 32 + lane] : Lay<Tl>::neg_inf();
      rd[j] = in ? blk_d[j * 32 + lane] : Lay<Tl>::neg_inf();
    }
    __syncwarp();
    bool last = false;
    if (lane == 0) last = stage_release_last(&S.cnt);
    last = __shfl_sync(FULL, last, 0);
    if (last && tma_next) issue_unit_load<Tl, R>(P, g, next, bar, smem_stage);
  } else {
    const char* tb = (const char*)P.target + ((size_t)trow * V + g.slice0()) * ES;
    const char* db = (const char*)P.draft + ((size_t)drow * V + g.slice0()) * ES;
    const int nv = nvec_of<Tl>(g), vb = g.vbeg(), ve = min(vb + 32 * g.rounds(), nv);
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int v = vb + j * 32 + lane;
      rt[j] = load_vec_direct<Tl>(tb, v, g.slen(), v < ve);
      rd[j] = load_vec_direct<Tl>(db, v, g.slen(), v < ve);
    }
  }

  const bool t_ok = T > 0.0f && T <= 3.0e38f;   // the losses need a sampling temperature
  const float c = t_ok ? fminf(__fdiv_rn(LOG2E_F, T), 3.0e38f) : 0.0f;

  // ---------------- pass A and the first exchange: row statistics
  MaxAcc<Tl> mx_t, mx_d;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    if (j == R - 1 && !last) break;
    mx_t.add(rt[j]);
    mx_d.add(rd[j]);
  }
  X1 mine;
  mine.m_t = warp_max_nan(mx_t.get());
  mine.m_d = warp_max_nan(mx_d.get());
  mine.i_t = 0; mine.i_d = 0;
  const u64 cc = pk(c, c);
  mine.ref_t = iref_of(mine.m_t, c);
  mine.ref_d = iref_of(mine.m_d, c);
  {
    const float rwt = mine.ref_t == NO_REF ? 0.0f : (float)mine.ref_t;
    const float rwd = mine.ref_d == NO_REF ? 0.0f : (float)mine.ref_d;
    mine.s_t = warp_sum_f32(rows_expsum<Tl, R>(rt, cc, pk(-rwt, -rwt), last));
    mine.s_d = warp_sum_f32(rows_expsum<Tl, R>(rd, cc, pk(-rwd, -rwd), last));
  }
  const int item = g.rank() * NWARP + warp;
  {
    const int set1 = n1 & 1;
    const uint32_t xbar = saddr(&S.xbar[set1]);
    if (tid == 0) mbar_expect_tx(xbar, (unsigned)g.items() * 32u);
    if (lane < (int)g.C()) st_async_x1(peer_addr(saddr(&S.x1[set1][item]), lane), mine, peer_addr(xbar, lane));
    const unsigned xpar = (unsigned)((n1 >> 1) & 1);
    ++n1;
    Merged& mg = S.mg[set1];
    if (warp == 0) {
      mbar_wait_cluster_bounded(xbar, xpar, P.flags);
      X1 z;
      z.m_t = -INFINITY; z.m_d = -INFINITY; z.s_t = 0.0f; z.s_d = 0.0f; z.i_t = 0; z.i_d = 0;
      z.ref_t = NO_REF; z.ref_d = NO_REF;
      const X1 ia = lane < g.items() ? S.x1[set1][lane] : z;
      const X1 ib = lane + 32 < g.items() ? S.x1[set1][lane + 32] : z;
      const float M_t = warp_max_nan(nanmax(ia.m_t, ib.m_t)), M_d = warp_max_nan(nanmax(ia.m_d, ib.m_d));
      const int IR_t = warp_max_s32(max(ia.ref_t, ib.ref_t)), IR_d = warp_max_s32(max(ia.ref_d, ib.ref_d));
      u64 st = add2(pk(ia.s_t * pow2_diff(ia.ref_t, IR_t), ia.s_d * pow2_diff(ia.ref_d, IR_d)),
                    pk(ib.s_t * pow2_diff(ib.ref_t, IR_t), ib.s_d * pow2_diff(ib.ref_d, IR_d)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float x, y;
        upk(st, x, y);
        st = add2(st, pk(__shfl_xor_sync(FULL, x, o), __shfl_xor_sync(FULL, y, o)));
      }
      float S_t, S_d;
      upk(st, S_t, S_d);
      const bool row_ok = t_ok && isfinite(M_t) && isfinite(M_d) && fabsf(M_t * c) < REF_LIMIT &&
                          fabsf(M_d * c) < REF_LIMIT && S_t > 0.0f && isfinite(S_t) && S_d > 0.0f && isfinite(S_d);
      if (lane == 0) {
        Merged m;
        m.S_t = S_t; m.S_d = S_d;
        m.R_t = IR_t == NO_REF ? 0.0f : (float)IR_t; m.R_d = IR_d == NO_REF ? 0.0f : (float)IR_d;
        m.r = row_ok ? S_t / S_d : 0.0f; m.IR_t = IR_t; m.status = row_ok ? 0 : ST_ROW; m.cont = 0; m.grab = -1;
        mg = m;
      }
      __syncwarp();
      merged_arrive();
    } else {
      merged_wait();
    }
  }
  const Merged M = S.mg[(n1 - 1) & 1];
  char* grow = (char*)P.grad + ((size_t)drow * V + g.slice0()) * ES;
  const int slen = g.slen(), vb = g.vbeg();
  if (M.status != 0) {   // invalid position: zero gradient, NaN loss
#pragma unroll
    for (int j = 0; j < R; ++j)
      if (j < g.rounds()) store_grad<Tl>(grow, vb + j * 32 + lane, slen, P.grad_vec, make_uint4(0u, 0u, 0u, 0u));
    if (tid == 0 && g.rank() == 0 && P.out_loss) P.out_loss[(size_t)b * k + ipos] = __int_as_float(0x7fc00000);
    return;
  }

  // ---------------- pass B: indicator bits and the two masses of this warp's range
  const u64 nrt = pk(-M.R_t, -M.R_t), nrd = pk(-M.R_d, -M.R_d), nr = pk(-M.r, -M.r);
  unsigned bits[NBW];
#pragma unroll
  for (int q = 0; q < NBW; ++q) bits[q] = 0u;
  u64 b1 = 0ull, b2 = 0ull;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    if (j == R - 1 && !last) break;
#pragma unroll
    for (int e = 0; e < EPV; e += 2) {
      const float t0 = Lay<Tl>::elem(rt[j], e), t1 = Lay<Tl>::elem(rt[j], e + 1);
      const float d0 = Lay<Tl>::elem(rd[j], e), d1 = Lay<Tl>::elem(rd[j], e + 1);
      float at0, at1, ad0, ad1;
      upk(fma2(pk(t0, t1), cc, nrt), at0, at1);
      upk(fma2(pk(d0, d1), cc, nrd), ad0, ad1);
      const float et0 = ex2(at0), et1 = ex2(at1), ed0 = ex2(ad0), ed1 = ex2(ad1);
      float y0, y1;
      upk(fma2(pk(ed0, ed1), nr, pk(et0, et1)), y0, y1);   // e_t - r e_d: > 0 exactly when q < p
      const bool i0 = y0 > 0.0f, i1 = y1 > 0.0f;
      const int pos = j * EPV + e;
      bits[pos >> 5] |= (i0 ? 1u : 0u) << (pos & 31);
      bits[(pos + 1) >> 5] |= (i1 ? 1u : 0u) << ((pos + 1) & 31);
      b1 = add2(b1, pk(i0 ? ed0 : 0.0f, i1 ? ed1 : 0.0f));
      b2 = add2(b2, pk(i0 ? 0.0f : et0, i1 ? 0.0f : et1));
    }
    if (j + 1 < R) fence_vec(rt[j + 1], rd[j + 1], b1);
  }
  X1 m2;
  {
    float x, y;
    upk(b1, x, y);
    m2.s_t = warp_sum_f32(x + y);
    upk(b2, x, y);
    m2.s_d = warp_sum_f32(x + y);
  }
  m2.m_t = 0.0f; m2.m_d = 0.0f; m2.i_t = 0; m2.i_d = 0; m2.ref_t = 0; m2.ref_d = 0;
  {
    const int set2 = n1 & 1;
    const uint32_t xbar = saddr(&S.xbar[set2]);
    if (tid == 0) mbar_expect_tx(xbar, (unsigned)g.items() * 32u);
    if (lane < (int)g.C()) st_async_x1(peer_addr(saddr(&S.x1[set2][item]), lane), m2, peer_addr(xbar, lane));
    const unsigned xpar = (unsigned)((n1 >> 1) & 1);
    ++n1;
    GradStat& gst = gs[set2];
    if (warp == 0) {
      mbar_wait_cluster_bounded(xbar, xpar, P.flags);
      float B1, B2;
      warp_sum_items(S.x1[set2], g.items(), B1, B2);
      const float beta = B1 / M.S_d;
      const float alpha = fmaf(M.r, B1, B2) / M.S_t;
      const int kind = P.loss_kind;
      const float w = P.weights ? P.weights[(size_t)b * k + ipos] : 1.0f;
      const float dl = kind == 0 ? -1.0f : -1.0f / alpha;
      if (lane == 0) {
        GradStat gv;
        gv.beta = beta;
        gv.K = w * dl / (T * M.S_d);
        gv.ok = 1; gv.pad = 0;
        gst = gv;
        if (g.rank() == 0 && P.out_loss) P.out_loss[(size_t)b * k + ipos] = kind == 0 ? 1.0f - alpha : -logf(alpha);
      }
      __syncwarp();
      merged_arrive();
    } else {
      merged_wait();
    }
  }
  const GradStat G = gs[(n1 - 1) & 1];

  // ---------------- pass C: the gradient of this warp's range of the draft row
  const float sel1 = G.K * (1.0f - G.beta), sel0 = -G.K * G.beta;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    if (j == R - 1 && !last) break;
    uint32_t wd[4];
#pragma unroll
    for (int e = 0; e < EPV; e += 2) {
      float ad0, ad1;
      upk(fma2(pk(Lay<Tl>::elem(rd[j], e), Lay<Tl>::elem(rd[j], e + 1)), cc, nrd), ad0, ad1);
      const int pos = j * EPV + e;
      const float s0 = (bits[pos >> 5] >> (pos & 31)) & 1u ? sel1 : sel0;
      const float s1 = (bits[(pos + 1) >> 5] >> ((pos + 1) & 31)) & 1u ? sel1 : sel0;
      float g0, g1;
      upk(mul2(pk(ex2(ad0), ex2(ad1)), pk(s0, s1)), g0, g1);
      if constexpr (sizeof(Tl) == 4) { wd[e] = __float_as_uint(g0); wd[e + 1] = __float_as_uint(g1); }
      else wd[e >> 1] = bf16x2_rn(g0, g1);   // rounded to nearest even
    }
    if (j < g.rounds())
      store_grad<Tl>(grow, vb + j * 32 + lane, slen, P.grad_vec, make_uint4(wd[0], wd[1], wd[2], wd[3]));
    if (j + 1 < R) {
      u64 dep = pk(__uint_as_float(wd[0]), __uint_as_float(wd[1]));
      fence_vec(rt[j + 1], rd[j + 1], dep);
    }
  }
}

template <typename Tl, int R>
__global__ void __launch_bounds__(NT, R <= 10 ? 2 : 1) sv_grad_kernel(const KParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ GradStat gs[2];
  Small& S = *reinterpret_cast<Small*>(smem);
  unsigned char* stage = smem + SMALL_BYTES;
  const int tid = threadIdx.x, warp = tid >> 5;
  Geo g;
  g.p = &P;
  const unsigned cid = cl_id(), ncl = cl_count();
  const unsigned B = (unsigned)P.B;
  const unsigned n_units = B * (unsigned)P.k;   // positions; below 2^31 (checked on the host)
  const uint32_t bar = saddr(&S.bar);
  const uint4* blk_t = reinterpret_cast<const uint4*>(stage) + (size_t)(0 * NWARP + warp) * R * 32;
  const uint4* blk_d = reinterpret_cast<const uint4*>(stage) + (size_t)(1 * NWARP + warp) * R * 32;
  if (P.tma) {
    uint4* st = reinterpret_cast<uint4*>(stage);
    for (int i = tid; i < 2 * NWARP * R * 32; i += NT) st[i] = Lay<Tl>::neg_inf();
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(saddr(&S.xbar[0]), 1);
    mbar_init(saddr(&S.xbar[1]), 1);
    S.cnt = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  cluster_sync_all();
  unsigned u = cid;
  Unit cur = pos_unit_of(u, B);
  if (P.tma && warp == 0 && u < n_units) issue_unit_load<Tl, R>(P, g, cur, bar, stage);
  unsigned phase = 0;
  int n1 = 0;
  for (; u < n_units; u += ncl, phase ^= 1u) {
    const bool has_next = u + ncl < n_units;
    const Unit next = pos_unit_of(u + ncl, B);
    grad_unit<Tl, R>(P, S, gs, blk_t, blk_d, g, cur, phase, n1, bar, stage, next, P.tma && has_next,
                     P.temperature[cur.b]);
    cur = next;
  }
  cluster_sync_all();
}

typedef void (*FusedFn)(const KParams);
typedef void (*FinalFn)(const FParams);
// Register rounds per thread.  Up to 10, two CTAs share an SM; at 16 and 20
// (the largest vocabularies) one CTA has the SM's register file to itself.
constexpr int R_CHOICES[] = {1, 2, 4, 6, 8, 10, 16, 20};
constexpr int N_R = 8;

template <typename Tl>
FusedFn pick_grad(int r) {
  switch (r) {
    case 1: return sv_grad_kernel<Tl, 1>;
    case 2: return sv_grad_kernel<Tl, 2>;
    case 4: return sv_grad_kernel<Tl, 4>;
    case 6: return sv_grad_kernel<Tl, 6>;
    case 8: return sv_grad_kernel<Tl, 8>;
    case 10: return sv_grad_kernel<Tl, 10>;
    case 16: return sv_grad_kernel<Tl, 16>;
    default: return sv_grad_kernel<Tl, 20>;
  }
}

template <typename Tl, int R>
void pick_r(FusedFn& f, FusedFn& fe, FusedFn& fl, FinalFn& g) {
  f = sv_fused_kernel<Tl, R, false, false>;
  fe = sv_fused_kernel<Tl, R, true, false>;
  fl = sv_fused_kernel<Tl, R, false, true>;
  g = sv_finalize_kernel<Tl, R>;
}
template <typename Tl>
void pick_kernels(int r, FusedFn& f, FusedFn& fe, FusedFn& fl, FinalFn& g) {
  switch (r) {
    case 1: pick_r<Tl, 1>(f, fe, fl, g); break;
    case 2: pick_r<Tl, 2>(f, fe, fl, g); break;
    case 4: pick_r<Tl, 4>(f, fe, fl, g); break;
    case 6: pick_r<Tl, 6>(f, fe, fl, g); break;
    case 8: pick_r<Tl, 8>(f, fe, fl, g); break;
    case 10: pick_r<Tl, 10>(f, fe, fl, g); break;
    case 16: pick_r<Tl, 16>(f, fe, fl, g); break;
    default: pick_r<Tl, 20>(f, fe, fl, g); break;
  }
}

}  // namespace

// ------------------------------------------------------------------ host side
// launch plan of one verification instance
struct VerifyPlan {
  size_t smem;        // dynamic shared memory (padded above the staged size when TMEM columns need it)
  int tmem_cols;      // TMEM columns per CTA (0: the instance uses none)
};

struct spec_verify_ctx {
  int device;
  int max_batch, k, V, dtype;
  unsigned flags;
  int C, Vs, R, rbase, rextra, n_clusters, tma_ok;
  size_t smem;               // dynamic shared memory of the fused kernels
  VerifyPlan plan_v, plan_ent, plan_lazy;   // the verification, entropy and lazy instances
  FusedFn kernel;
  FusedFn kernel_ent;        // the same kernel that also writes row entropies
  int n_clusters_ent;
  FusedFn kernel_grad;       // loss-gradient kernel
  int n_clusters_grad;
  FusedFn kernel_lazy;       // lazy verification (each chain up to its first rejection)
  int* ws_grab;              // lazy verification: chain hand-out counter
  int n_clusters_lazy;
  FinalFn finalize;
  int32_t* ws_acc;
  int32_t* ws_y;
  UnitStat* ws_stat;
  float* ws_w;
  float* ws_p;
  int* d_flags;
  // host staging (SV_FLAG_HOST_STAGING)
  void* st_target;
  void* st_draft;
  int32_t* st_tokens;
  float* st_temp;
  float* st_unif;
  int32_t* st_out_tokens;
  int32_t* st_out_tau;
  float* st_out_p;
  float* st_out_q;
  float* st_out_tv;
  // kernel timing (SV_FLAG_KERNEL_TIMING)
  cudaEvent_t* ev;   // 2 * TIMING_RING events
  int ev_n;          // calls recorded since the last read
};

static constexpr int TIMING_RING = 4096;

// Dynamic shared memory of one CTA with R register rounds: the bookkeeping
// area, and the bulk-copy stage (two rows of NWARP blocks of R*32 vectors).
// Kernels with plain loads use only the bookkeeping area.
static size_t smem_bytes(int R, bool tma) { return SMALL_BYTES + (tma ? 2 * (size_t)NWARP * R * 32 * 16 : 0); }

// The opt-in limit is a property of the kernel, shared by every handle and
// plan that launches it: set it to the largest size any launch of this R asks
// for (the staged one), so that opening a handle with plain loads never
// lowers it under a live handle that stages.
static bool set_smem_limit(FusedFn f, int R) {
  return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes(R, true)) == cudaSuccess;
}

// Never launched: the occupancy calculation reports the number of clusters of
// C CTAs that fit when each SM holds a given number of CTAs, set through this
// kernel's dynamic shared memory.
__global__ void sv_cluster_fit_kernel(int*) {}

// Launch plan of the verification instance (the kernel that keeps target
// exponentials in TMEM): dynamic shared memory, TMEM columns per CTA, and the
// number of co-resident clusters.
//  - Each CTA allocates the power of 2 at or above the 2 EPV R columns its
//    warps use (two warps per lane quarter) and holds them for the whole
//    kernel.  The CTAs an SM holds at once must fit in its 512 columns, or one
//    could wait for columns that its own cluster's progress is needed to free;
//    the shared-memory request is padded until the SM's other limits allow no
//    more CTAs than that.
//  - The occupancy calculation assumes that a kernel using TMEM owns the SM
//    (it reports one CTA per SM), while the hardware schedules such CTAs by
//    registers, shared memory and threads like any other (measured: two CTAs
//    of 256 columns on every SM).  So CTAs per SM are counted here from those
//    limits, and the number of clusters that fit with that many CTAs per SM is
//    taken from a stand-in kernel without TMEM.
static int plan_verify(FusedFn f, int R, int epv, int C, size_t smem0, size_t smem_staged, VerifyPlan* plan,
                       int* n_clusters) {
  int dev = 0, optin = 0, sm_smem = 0, sm_regs = 0, sm_thr = 0, sm_blocks = 0, reserved = 0;
  cudaFuncAttributes fa;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sm_regs, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sm_thr, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sm_blocks, cudaDevAttrMaxBlocksPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
      cudaFuncGetAttributes(&fa, f) != cudaSuccess)
    return SV_ERR_CUDA;
  optin -= (int)fa.sharedSizeBytes;   // the limit covers dynamic shared memory only
  const bool uses = tmem_used(epv, R);
  int need = 0;   // warps 0..3 and 4..7 each take tmem_cols_per_warp columns
  if (uses) {
    need = 32;
    while (need < 2 * tmem_cols_per_warp(epv, R)) need <<= 1;
  }
  const int tmem_ctas = uses ? 512 / need : 1 << 30;
  // registers are allocated per warp in multiples of 256
  const long long regs_cta = (long long)((fa.numRegs * 32 + 255) / 256 * 256) * (NT / 32);
  size_t sm = smem0;
  // A TMEM instance must leave no room on an SM for a third such CTA of any
  // of these kernels (a second one at 512 columns): by its registers, as
  // every one compiled here does, or else by shared memory.
  if (uses && regs_cta * (512 / need + 1) <= sm_regs) {
    const size_t floor_smem = (size_t)(sm_smem / (512 / need + 1) - reserved - (int)fa.sharedSizeBytes + 1);
    if (sm < floor_smem) sm = floor_smem;
  }
  int ctas = 0;
  for (;;) {
    const long long by_smem = (long long)sm_smem / ((long long)sm + fa.sharedSizeBytes + reserved);
    long long c = sm_regs / regs_cta;
    c = c < by_smem ? c : by_smem;
    c = c < sm_thr / NT ? c : sm_thr / NT;
    c = c < sm_blocks ? c : sm_blocks;
    if (c <= 0) return SV_ERR_SIZE;
    if (c <= tmem_ctas) { ctas = (int)c; break; }
    sm += 4096;   // fewer CTAs per SM
    if (sm > (size_t)optin) return SV_ERR_SIZE;
  }
  // the opt-in limit is shared by every handle of this kernel: raised to the
  // largest request any plan makes (the staged one, or a padded one), never lowered
  const size_t lim = sm > smem_staged ? sm : smem_staged;
  if ((int)lim > fa.maxDynamicSharedSizeBytes &&
      cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lim) != cudaSuccess)
    return SV_ERR_CUDA;
  const int fit_smem = sm_smem / ctas - reserved;   // the stand-in then holds `ctas` CTAs per SM
  if (cudaFuncSetAttribute(sv_cluster_fit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, fit_smem) != cudaSuccess)
    return SV_ERR_CUDA;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)C, 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)fit_smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int per_sm = 0, n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sv_cluster_fit_kernel, NT, (size_t)fit_smem) != cudaSuccess ||
      per_sm != ctas || cudaOccupancyMaxActiveClusters(&n, sv_cluster_fit_kernel, &cfg) != cudaSuccess || n <= 0)
    return SV_ERR_CUDA;
  plan->smem = sm;
  plan->tmem_cols = need;
  *n_clusters = n;
  return SV_OK;
}

static void free_ctx(spec_verify_ctx* h) {
  if (!h) return;
  void* ptrs[] = {h->ws_acc, h->ws_y, h->ws_stat, h->ws_w, h->ws_p, h->d_flags, h->ws_grab, h->st_target, h->st_draft, h->st_tokens, h->st_temp,
                  h->st_unif, h->st_out_tokens, h->st_out_tau, h->st_out_p, h->st_out_q, h->st_out_tv};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  if (h->ev) {
    for (int i = 0; i < 2 * TIMING_RING; ++i)
      if (h->ev[i]) cudaEventDestroy(h->ev[i]);
    free(h->ev);
  }
  free(h);
}

// Units of one verification call: the k verified positions of every chain,
// then the bonus rows two to a unit.
static long long verify_units(int batch, int k) { return (long long)batch * k + (batch + 1) / 2; }

static int launch_fused(spec_verify_ctx* h, const KParams& P, long long units, cudaStream_t s, bool grad = false,
                        bool lazy = false) {
  const bool ent = P.out_ent_t || P.out_ent_d;
  const int ncl = grad ? h->n_clusters_grad : lazy ? h->n_clusters_lazy : ent ? h->n_clusters_ent : h->n_clusters;
  const int grid_clusters = (int)(units < ncl ? units : ncl);
  if (grid_clusters <= 0) return SV_OK;
  const bool timed = h->ev && h->ev_n < TIMING_RING;
  if (timed && cudaEventRecord(h->ev[2 * h->ev_n], s) != cudaSuccess) return SV_ERR_CUDA;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)(grid_clusters * h->C), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  const VerifyPlan& vp = lazy ? h->plan_lazy : ent ? h->plan_ent : h->plan_v;
  cfg.dynamicSmemBytes = grad ? h->smem : vp.smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)h->C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  KParams Q = P;
  Q.tmem_cols = grad ? 0 : vp.tmem_cols;
  if (cudaLaunchKernelEx(&cfg, grad ? h->kernel_grad : lazy ? h->kernel_lazy : ent ? h->kernel_ent : h->kernel, Q) !=
      cudaSuccess)
    return SV_ERR_CUDA;
  if (timed) {
    if (cudaEventRecord(h->ev[2 * h->ev_n + 1], s) != cudaSuccess) return SV_ERR_CUDA;
    h->ev_n++;
  }
  return SV_OK;
}

static int launch_finalize(spec_verify_ctx* h, const KParams& P, const int32_t* tokens, int32_t* out_tokens,
                           int32_t* out_tau, cudaStream_t s, bool lazy = false) {
  FParams F;
  memset(&F, 0, sizeof F);
  F.target = P.target; F.draft = P.draft; F.tokens = tokens; F.uniforms = P.uniforms;
  F.ws_acc = P.ws_acc; F.ws_y = P.ws_y; F.ws_stat = P.ws_stat; F.ws_w = P.ws_w; F.ws_p = P.ws_p;
  F.out_tokens = out_tokens; F.out_tau = out_tau; F.out_tv = P.out_tv; F.flags = P.flags;
  F.B = P.B; F.k = P.k; F.V = P.V; F.Vs = P.Vs; F.rbase = P.rbase; F.rextra = P.rextra; F.items = h->C * NWARP; F.vec16 = P.tma || P.vec16;
  F.tv_only = P.tv_only;
  F.lazy = lazy ? 1 : 0;
  h->finalize<<<(P.B + 7) / 8, 256, 0, s>>>(F);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

// ---------------------------------------------------- allocation-free entry
// spec_verify_noalloc keeps its workspace in this file-scope device array
// instead of memory from cudaMalloc.  Every GPU that loads the library holds
// one copy until the process exits.  Host code must not use the array's name
// as a device address: the address is looked up once per device with
// cudaGetSymbolAddress and passed to the kernels.
constexpr size_t NOALLOC_BYTES = (size_t)SV_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

namespace {
struct NoallocDevice {       // per-device set-up, done by the first call on that device
  bool ready;
  unsigned char* scratch;    // device address of g_noalloc_scratch
};
constexpr int NOALLOC_MAX_DEVICES = 64;
NoallocDevice g_noalloc_dev[NOALLOC_MAX_DEVICES];
struct NoallocPlan {         // launch geometry cached per (device, k, V, dtype)
  bool used;
  int device, k, V, dtype;
  spec_verify_ctx plan;      // only the geometry and kernel fields are filled
};
constexpr int NOALLOC_PLANS = 32;
NoallocPlan g_noalloc_plans[NOALLOC_PLANS];
std::mutex g_noalloc_lock;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Byte offsets of the workspace arrays inside the scratch array.
struct NoallocLayout {
  size_t flags, acc, y, stat, w, p, total;
};
NoallocLayout noalloc_layout(size_t B, size_t k) {
  NoallocLayout L;
  L.flags = 0;
  L.acc = align256(L.flags + 4 * sizeof(int));
  L.y = align256(L.acc + B * k * sizeof(int32_t));
  L.stat = align256(L.y + B * (k + 1) * sizeof(int32_t));
  L.w = align256(L.stat + B * (k + 1) * sizeof(UnitStat));
  L.p = align256(L.w + B * (k + 1) * ITEMS_MAX * sizeof(float));
  L.total = L.p + B * (k + 1) * ITEMS_MAX * sizeof(float);
  return L;
}

// Geometry, kernels and occupancy for (k, V, dtype) on the current device;
// the same choices spec_verify_init makes.  Allocates nothing.
int noalloc_plan(int device, int k, int vocab, int dtype, spec_verify_ctx& out) {
  for (int i = 0; i < NOALLOC_PLANS; ++i) {
    const NoallocPlan& c = g_noalloc_plans[i];
    if (c.used && c.device == device && c.k == k && c.V == vocab && c.dtype == dtype) {
      out = c.plan;
      return SV_OK;
    }
  }
  spec_verify_ctx h;
  memset(&h, 0, sizeof h);
  const int es = dtype == SV_FP32 ? 4 : 2;
  const int epv = 16 / es;
  int C = 1;
  for (int c = CMAX; c >= 1; c >>= 1) {
    const long long vs = ((long long)(vocab + c - 1) / c + epv - 1) / epv * epv;
    if (vs >= (long long)NT * epv || c == 1) { C = c; break; }
  }
  const long long Vs = ((long long)(vocab + C - 1) / C + epv - 1) / epv * epv;
  const long long nvec = Vs / epv;
  const long long nrounds = (nvec + 31) / 32;   // per CTA slice, split over the warps
  const long long rbase = nrounds / NWARP, rextra = nrounds % NWARP;
  const long long r_need = rbase + (rextra > 0 ? 1 : 0);
  int R = -1;
  for (int i = 0; i < N_R; ++i)
    if (R_CHOICES[i] >= r_need) { R = R_CHOICES[i]; break; }
  if (R < 0) return SV_ERR_SIZE;
  h.device = device; h.k = k; h.V = vocab; h.dtype = dtype;
  h.C = C; h.Vs = (int)Vs; h.R = R; h.rbase = (int)rbase; h.rextra = (int)rextra;
  h.tma_ok = ((size_t)vocab * es) % 16 == 0;
  h.smem = smem_bytes(R, h.tma_ok);
  if (dtype == SV_FP32) pick_kernels<float>(R, h.kernel, h.kernel_ent, h.kernel_lazy, h.finalize);
  else pick_kernels<__nv_bfloat16>(R, h.kernel, h.kernel_ent, h.kernel_lazy, h.finalize);
  const int rc = plan_verify(h.kernel, R, epv, C, h.smem, smem_bytes(R, true), &h.plan_v, &h.n_clusters);
  if (rc != SV_OK) {
    cudaGetLastError();
    return rc;
  }
  for (int i = 0; i < NOALLOC_PLANS; ++i) {
    if (!g_noalloc_plans[i].used) {
      g_noalloc_plans[i].used = true;
      g_noalloc_plans[i].device = device; g_noalloc_plans[i].k = k; g_noalloc_plans[i].V = vocab;
      g_noalloc_plans[i].dtype = dtype;
      g_noalloc_plans[i].plan = h;
      break;
    }
  }
  out = h;
  return SV_OK;
}
}  // namespace

extern "C" {

const char* spec_verify_strerror(int code) {
  switch (code) {
    case SV_OK: return "ok";
    case SV_ERR_ARG: return "invalid argument";
    case SV_ERR_DTYPE: return "unsupported logit dtype";
    case SV_ERR_SIZE: return "k or vocabulary size outside the supported range";
    case SV_ERR_CUDA: return "CUDA runtime error";
    case SV_ERR_ALLOC: return "allocation failed";
    case SV_ERR_DATA: return "invalid chains (token out of range, bad temperature or non-finite logits)";
    case SV_ERR_TIMEOUT: return "a bounded device wait expired";
    default: return "unknown status";
  }
}

int spec_verify_init(spec_verify_t* out, int max_batch, int k, int vocab, int logit_dtype, unsigned flags) {
  if (!out) return SV_ERR_ARG;
  *out = nullptr;
  if (max_batch < 0) return SV_ERR_ARG;
  if (logit_dtype != SV_FP32 && logit_dtype != SV_BF16) return SV_ERR_DTYPE;
  if (k < 1 || k > 31 || vocab < 1) return SV_ERR_SIZE;
  if ((long long)max_batch * (k + 1) >= (1LL << 31)) return SV_ERR_SIZE;   // units are counted in 32 bits
  const int es = logit_dtype == SV_FP32 ? 4 : 2;
  const int epv = 16 / es;
  // cluster size: the largest of 8/4/2/1 that still gives each CTA a full round
  int C = 1;
  for (int c = CMAX; c >= 1; c >>= 1) {
    const long long vs = ((long long)(vocab + c - 1) / c + epv - 1) / epv * epv;
    if (vs >= (long long)NT * epv || c == 1) { C = c; break; }
  }
  const long long Vs = ((long long)(vocab + C - 1) / C + epv - 1) / epv * epv;
  const long long nvec = Vs / epv;
  const long long nrounds = (nvec + 31) / 32;   // per CTA slice, split over the warps
  const long long rbase = nrounds / NWARP, rextra = nrounds % NWARP;
  const long long r_need = rbase + (rextra > 0 ? 1 : 0);
  int R = -1;
  for (int i = 0; i < N_R; ++i)
    if (R_CHOICES[i] >= r_need) { R = R_CHOICES[i]; break; }
  if (R < 0) return SV_ERR_SIZE;

  spec_verify_ctx* h = (spec_verify_ctx*)calloc(1, sizeof(spec_verify_ctx));
  if (!h) return SV_ERR_ALLOC;
  if (cudaGetDevice(&h->device) != cudaSuccess) { free(h); return SV_ERR_CUDA; }
  h->max_batch = max_batch; h->k = k; h->V = vocab; h->dtype = logit_dtype; h->flags = flags;
  h->C = C; h->Vs = (int)Vs; h->R = R; h->rbase = (int)rbase; h->rextra = (int)rextra;
  h->tma_ok = ((size_t)vocab * es) % 16 == 0 && !(flags & SV_FLAG_NO_TMA);
  h->smem = smem_bytes(R, h->tma_ok);
  if (logit_dtype == SV_FP32) pick_kernels<float>(R, h->kernel, h->kernel_ent, h->kernel_lazy, h->finalize);
  else pick_kernels<__nv_bfloat16>(R, h->kernel, h->kernel_ent, h->kernel_lazy, h->finalize);
  h->kernel_grad = logit_dtype == SV_FP32 ? pick_grad<float>(R) : pick_grad<__nv_bfloat16>(R);
  if (!set_smem_limit(h->kernel_grad, R)) {
    free_ctx(h);
    return SV_ERR_CUDA;
  }
  {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)C, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = h->smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int ng = 0;
    int rc = plan_verify(h->kernel, R, epv, C, h->smem, smem_bytes(R, true), &h->plan_v, &h->n_clusters);
    if (rc == SV_OK)
      rc = plan_verify(h->kernel_ent, R, epv, C, h->smem, smem_bytes(R, true), &h->plan_ent, &h->n_clusters_ent);
    if (rc == SV_OK)
      rc = plan_verify(h->kernel_lazy, R, epv, C, h->smem, smem_bytes(R, true), &h->plan_lazy, &h->n_clusters_lazy);
    if (rc != SV_OK) {
      cudaGetLastError();
      free_ctx(h);
      return rc;
    }
    if (cudaOccupancyMaxActiveClusters(&ng, h->kernel_grad, &cfg) != cudaSuccess || ng <= 0) {
      cudaGetLastError();
      free_ctx(h);
      return SV_ERR_CUDA;
    }
    h->n_clusters_grad = ng;
  }
  const size_t mb = (size_t)(max_batch > 0 ? max_batch : 1);
  bool ok = cudaMalloc(&h->ws_acc, mb * k * sizeof(int32_t)) == cudaSuccess &&
            cudaMalloc(&h->ws_y, mb * (k + 1) * sizeof(int32_t)) == cudaSuccess &&
            cudaMalloc(&h->ws_stat, mb * (k + 1) * sizeof(UnitStat)) == cudaSuccess &&
            cudaMalloc(&h->ws_w, mb * (k + 1) * ITEMS_MAX * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&h->ws_p, mb * (k + 1) * ITEMS_MAX * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&h->d_flags, 4 * sizeof(int)) == cudaSuccess &&
            cudaMalloc(&h->ws_grab, sizeof(int)) == cudaSuccess;
  if (ok && (flags & SV_FLAG_HOST_STAGING)) {
    const size_t rowb = (size_t)vocab * es;
    ok = cudaMalloc(&h->st_target, mb * (k + 1) * rowb) == cudaSuccess &&
         cudaMalloc(&h->st_draft, mb * k * rowb) == cudaSuccess &&
         cudaMalloc(&h->st_tokens, mb * k * sizeof(int32_t)) == cudaSuccess &&
         cudaMalloc(&h->st_temp, mb * sizeof(float)) == cudaSuccess &&
         cudaMalloc(&h->st_unif, mb * (k + 1) * sizeof(float)) == cudaSuccess &&
         cudaMalloc(&h->st_out_tokens, mb * (k + 1) * sizeof(int32_t)) == cudaSuccess &&
         cudaMalloc(&h->st_out_tau, mb * sizeof(int32_t)) == cudaSuccess &&
         cudaMalloc(&h->st_out_p, mb * k * sizeof(float)) == cudaSuccess &&
         cudaMalloc(&h->st_out_q, mb * k * sizeof(float)) == cudaSuccess &&
         cudaMalloc(&h->st_out_tv, mb * k * sizeof(float)) == cudaSuccess;
  }
  if (!ok) {
    cudaGetLastError();
    free_ctx(h);
    return SV_ERR_ALLOC;
  }
  if (cudaMemset(h->d_flags, 0, 4 * sizeof(int)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    free_ctx(h);
    return SV_ERR_CUDA;
  }
  if (flags & SV_FLAG_KERNEL_TIMING) {
    h->ev = (cudaEvent_t*)calloc(2 * TIMING_RING, sizeof(cudaEvent_t));
    if (!h->ev) { free_ctx(h); return SV_ERR_ALLOC; }
    for (int i = 0; i < 2 * TIMING_RING; ++i)
      if (cudaEventCreate(&h->ev[i]) != cudaSuccess) { free_ctx(h); return SV_ERR_CUDA; }
  }
  *out = h;
  return SV_OK;
}

static bool al4(const void* p) { return ((uintptr_t)p & 3u) == 0; }
static bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int spec_verify(spec_verify_t h, int batch, const void* target_logits, const void* draft_logits,
                const int32_t* draft_tokens, const float* temperature, const float* uniforms,
                int32_t* out_tokens, int32_t* out_tau, float* out_p_draft, float* out_q_draft, float* out_tv,
                void* cuda_stream) {
  return spec_verify_ex(h, batch, target_logits, draft_logits, draft_tokens, temperature, uniforms, out_tokens, out_tau,
                        out_p_draft, out_q_draft, out_tv, nullptr, nullptr, cuda_stream);
}

// The verification step.  bulk_ok = false keeps the kernels off bulk copies
// (logits in host memory, read in place).
static int verify_impl(spec_verify_t h, int batch, const void* target_logits, const void* draft_logits,
                       const int32_t* draft_tokens, const float* temperature, const float* uniforms,
                       int32_t* out_tokens, int32_t* out_tau, float* out_p_draft, float* out_q_draft, float* out_tv,
                       float* out_entropy_target, float* out_entropy_draft, void* cuda_stream, bool bulk_ok) {
  if (!h || batch < 0 || batch > h->max_batch) return SV_ERR_ARG;
  if (batch == 0) return SV_OK;
  if (!target_logits || !draft_logits || !draft_tokens || !temperature || !uniforms || !out_tokens || !out_tau)
    return SV_ERR_ARG;
  const int es = h->dtype == SV_FP32 ? 4 : 2;
  if (((uintptr_t)target_logits % es) || ((uintptr_t)draft_logits % es)) return SV_ERR_ARG;
  if (!al4(draft_tokens) || !al4(temperature) || !al4(uniforms) || !al4(out_tokens) || !al4(out_tau) ||
      !al4(out_p_draft) || !al4(out_q_draft) || !al4(out_tv) || !al4(out_entropy_target) || !al4(out_entropy_draft))
    return SV_ERR_ARG;
  if ((out_entropy_target == nullptr) != (out_entropy_draft == nullptr)) return SV_ERR_ARG;
  cudaStream_t s = (cudaStream_t)cuda_stream;
  KParams P;
  memset(&P, 0, sizeof P);
  P.target = target_logits; P.draft = draft_logits; P.tokens = draft_tokens; P.temperature = temperature;
  P.uniforms = uniforms; P.out_p = out_p_draft; P.out_q = out_q_draft; P.out_tv = out_tv;
  P.out_ent_t = out_entropy_target; P.out_ent_d = out_entropy_draft;
  P.ws_acc = h->ws_acc; P.ws_y = h->ws_y; P.ws_stat = h->ws_stat; P.ws_w = h->ws_w; P.ws_p = h->ws_p;
  P.flags = h->d_flags;
  P.B = batch; P.k = h->k; P.V = h->V; P.Vs = h->Vs; P.rbase = h->rbase; P.rextra = h->rextra;
  P.units_per_chain = h->k + 1; P.tv_only = 0;
  P.vec16 = h->tma_ok && al16(target_logits) && al16(draft_logits);
  P.tma = bulk_ok && P.vec16;
  int rc = launch_fused(h, P, verify_units(batch, h->k), s);
  if (rc != SV_OK) return rc;
  return launch_finalize(h, P, draft_tokens, out_tokens, out_tau, s);
}

int spec_verify_ex(spec_verify_t h, int batch, const void* target_logits, const void* draft_logits,
                   const int32_t* draft_tokens, const float* temperature, const float* uniforms,
                   int32_t* out_tokens, int32_t* out_tau, float* out_p_draft, float* out_q_draft, float* out_tv,
                   float* out_entropy_target, float* out_entropy_draft, void* cuda_stream) {
  return verify_impl(h, batch, target_logits, draft_logits, draft_tokens, temperature, uniforms, out_tokens, out_tau,
                     out_p_draft, out_q_draft, out_tv, out_entropy_target, out_entropy_draft, cuda_stream, true);
}

int spec_verify_lazy(spec_verify_t h, int batch, const void* target_logits, const void* draft_logits,
                     const int32_t* draft_tokens, const float* temperature, const float* uniforms,
                     int32_t* out_tokens, int32_t* out_tau, void* cuda_stream) {
  if (!h || batch < 0 || batch > h->max_batch) return SV_ERR_ARG;
  if (batch == 0) return SV_OK;
  if (!target_logits || !draft_logits || !draft_tokens || !temperature || !uniforms || !out_tokens || !out_tau)
    return SV_ERR_ARG;
  const int es = h->dtype == SV_FP32 ? 4 : 2;
  if (((uintptr_t)target_logits % es) || ((uintptr_t)draft_logits % es)) return SV_ERR_ARG;
  if (!al4(draft_tokens) || !al4(temperature) || !al4(uniforms) || !al4(out_tokens) || !al4(out_tau)) return SV_ERR_ARG;
  cudaStream_t s = (cudaStream_t)cuda_stream;
  KParams P;
  memset(&P, 0, sizeof P);
  P.target = target_logits; P.draft = draft_logits; P.tokens = draft_tokens; P.temperature = temperature;
  P.uniforms = uniforms;
  P.ws_acc = h->ws_acc; P.ws_y = h->ws_y; P.ws_stat = h->ws_stat; P.ws_w = h->ws_w; P.ws_p = h->ws_p;
  P.flags = h->d_flags;
  P.B = batch; P.k = h->k; P.V = h->V; P.Vs = h->Vs; P.rbase = h->rbase; P.rextra = h->rextra;
  P.units_per_chain = h->k + 1; P.tv_only = 0;
  P.tma = h->tma_ok && al16(target_logits) && al16(draft_logits);
  P.vec16 = P.tma;
  P.ws_grab = h->ws_grab;
  if (cudaMemsetAsync(h->ws_grab, 0, sizeof(int), s) != cudaSuccess) return SV_ERR_CUDA;
  const int rc = launch_fused(h, P, batch, s, false, true);
  if (rc != SV_OK) return rc;
  return launch_finalize(h, P, draft_tokens, out_tokens, out_tau, s, true);
}

int spec_verify_noalloc(int batch, int k, int vocab, int logit_dtype, const void* target_logits,
                        const void* draft_logits, const int32_t* draft_tokens, const float* temperature,
                        const float* uniforms, int32_t* out_tokens, int32_t* out_tau, float* out_p_draft,
                        float* out_q_draft, float* out_tv, void* cuda_stream) {
  if (batch < 0) return SV_ERR_ARG;
  if (logit_dtype != SV_FP32 && logit_dtype != SV_BF16) return SV_ERR_DTYPE;
  if (k < 1 || k > 31 || vocab < 1) return SV_ERR_SIZE;
  const NoallocLayout L = noalloc_layout((size_t)batch, (size_t)k);
  if (L.total > NOALLOC_BYTES) return SV_ERR_SIZE;
  if (batch == 0) return SV_OK;
  if (!target_logits || !draft_logits || !draft_tokens || !temperature || !uniforms || !out_tokens || !out_tau)
    return SV_ERR_ARG;
  const int es = logit_dtype == SV_FP32 ? 4 : 2;
  if (((uintptr_t)target_logits % es) || ((uintptr_t)draft_logits % es)) return SV_ERR_ARG;
  if (!al4(draft_tokens) || !al4(temperature) || !al4(uniforms) || !al4(out_tokens) || !al4(out_tau) ||
      !al4(out_p_draft) || !al4(out_q_draft) || !al4(out_tv))
    return SV_ERR_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return SV_ERR_CUDA;
  if (device < 0 || device >= NOALLOC_MAX_DEVICES) return SV_ERR_ARG;
  spec_verify_ctx h;
  unsigned char* scratch = nullptr;
  {
    std::lock_guard<std::mutex> guard(g_noalloc_lock);
    NoallocDevice& d = g_noalloc_dev[device];
    if (!d.ready) {   // once per device, with that device current
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return SV_ERR_CUDA;
      }
      d.scratch = (unsigned char*)ptr;
      d.ready = true;
    }
    scratch = d.scratch;
    const int rc = noalloc_plan(device, k, vocab, logit_dtype, h);
    if (rc != SV_OK) return rc;
  }
  cudaStream_t s = (cudaStream_t)cuda_stream;
  int* flags = (int*)(scratch + L.flags);
  if (cudaMemsetAsync(flags, 0, 4 * sizeof(int), s) != cudaSuccess) return SV_ERR_CUDA;   // counters start at zero
  KParams P;
  memset(&P, 0, sizeof P);
  P.target = target_logits; P.draft = draft_logits; P.tokens = draft_tokens; P.temperature = temperature;
  P.uniforms = uniforms; P.out_p = out_p_draft; P.out_q = out_q_draft; P.out_tv = out_tv;
  P.ws_acc = (int32_t*)(scratch + L.acc); P.ws_y = (int32_t*)(scratch + L.y);
  P.ws_stat = (UnitStat*)(scratch + L.stat); P.ws_w = (float*)(scratch + L.w); P.ws_p = (float*)(scratch + L.p);
  P.flags = flags;
  P.B = batch; P.k = k; P.V = vocab; P.Vs = h.Vs; P.rbase = h.rbase; P.rextra = h.rextra;
  P.units_per_chain = k + 1; P.tv_only = 0;
  P.tma = h.tma_ok && al16(target_logits) && al16(draft_logits);
  P.vec16 = P.tma;
  int rc = launch_fused(&h, P, verify_units(batch, k), s);
  if (rc != SV_OK) return rc;
  return launch_finalize(&h, P, draft_tokens, out_tokens, out_tau, s);
}

int spec_verify_tv(spec_verify_t h, int batch, const void* target_logits, const void* draft_logits,
                   const float* temperature, float* out_tv, void* cuda_stream) {
  if (!h || batch < 0 || batch > h->max_batch) return SV_ERR_ARG;
  if (batch == 0) return SV_OK;
  if (!target_logits || !draft_logits || !temperature || !out_tv) return SV_ERR_ARG;
  const int es = h->dtype == SV_FP32 ? 4 : 2;
  if (((uintptr_t)target_logits % es) || ((uintptr_t)draft_logits % es)) return SV_ERR_ARG;
  if (!al4(temperature) || !al4(out_tv)) return SV_ERR_ARG;
  KParams P;
  memset(&P, 0, sizeof P);
  P.target = target_logits; P.draft = draft_logits; P.temperature = temperature; P.out_tv = out_tv;
  P.ws_acc = h->ws_acc; P.ws_y = h->ws_y; P.ws_stat = h->ws_stat; P.ws_w = h->ws_w; P.ws_p = h->ws_p;
  P.flags = h->d_flags;
  P.B = batch; P.k = h->k; P.V = h->V; P.Vs = h->Vs; P.rbase = h->rbase; P.rextra = h->rextra;
  P.units_per_chain = h->k; P.tv_only = 1;
  P.tma = h->tma_ok && al16(target_logits) && al16(draft_logits);
  P.vec16 = P.tma;
  cudaStream_t s = (cudaStream_t)cuda_stream;
  int rc = launch_fused(h, P, (long long)batch * h->k, s);
  if (rc != SV_OK) return rc;
  return launch_finalize(h, P, nullptr, nullptr, nullptr, s);
}

int spec_verify_loss_grad(spec_verify_t h, int batch, const void* target_logits, const void* draft_logits,
                          const float* temperature, int loss_kind, const float* weights, float* out_loss,
                          void* grad_draft, void* cuda_stream) {
  if (!h || batch < 0 || batch > h->max_batch) return SV_ERR_ARG;
  if (loss_kind != SV_LOSS_TV && loss_kind != SV_LOSS_OVERLAP) return SV_ERR_ARG;
  if (batch == 0) return SV_OK;
  if (!target_logits || !draft_logits || !temperature || !grad_draft) return SV_ERR_ARG;
  const int es = h->dtype == SV_FP32 ? 4 : 2;
  if (((uintptr_t)target_logits % es) || ((uintptr_t)draft_logits % es) || ((uintptr_t)grad_draft % es)) return SV_ERR_ARG;
  if (!al4(temperature) || !al4(weights) || !al4(out_loss)) return SV_ERR_ARG;
  KParams P;
  memset(&P, 0, sizeof P);
  P.target = target_logits; P.draft = draft_logits; P.temperature = temperature;
  P.weights = weights; P.out_loss = out_loss; P.grad = grad_draft; P.loss_kind = loss_kind;
  P.flags = h->d_flags;
  P.B = batch; P.k = h->k; P.V = h->V; P.Vs = h->Vs; P.rbase = h->rbase; P.rextra = h->rextra;
  P.units_per_chain = h->k; P.tv_only = 1;
  P.tma = h->tma_ok && al16(target_logits) && al16(draft_logits);
  P.vec16 = P.tma;
  P.grad_vec = ((size_t)h->V * es) % 16 == 0 && al16(grad_draft);
  return launch_fused(h, P, (long long)batch * h->k, (cudaStream_t)cuda_stream, true);
}

// The device address of host memory the device can read directly (page-locked
// memory on a system with unified addressing), else null.
static const void* device_view(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

int spec_verify_host(spec_verify_t h, int batch, const void* host_target_logits, const void* host_draft_logits,
                     const int32_t* host_draft_tokens, const float* host_temperature, const float* host_uniforms,
                     int32_t* host_out_tokens, int32_t* host_out_tau, float* host_out_p_draft,
                     float* host_out_q_draft, float* host_out_tv, void* cuda_stream) {
  if (!h || !(h->flags & SV_FLAG_HOST_STAGING) || batch < 0 || batch > h->max_batch) return SV_ERR_ARG;
  if (batch == 0) return SV_OK;
  if (!host_target_logits || !host_draft_logits || !host_draft_tokens || !host_temperature || !host_uniforms ||
      !host_out_tokens || !host_out_tau)
    return SV_ERR_ARG;
  cudaStream_t s = (cudaStream_t)cuda_stream;
  const int es = h->dtype == SV_FP32 ? 4 : 2;
  const size_t B = (size_t)batch, k = (size_t)h->k, rowb = (size_t)h->V * es;
  const cudaMemcpyKind H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;
  // Logits in page-locked host memory that the device addresses directly are
  // read in place by the kernels, over the host link, with 16-byte loads (no
  // bulk copies from host memory).  Other host memory is copied into the
  // device staging buffers first.  Either way every logit crosses the link
  // once; reading in place saves the separate copy before the kernels.
  const void* dev_t = device_view(host_target_logits);
  const void* dev_d = device_view(host_draft_logits);
  const bool in_place = dev_t && dev_d;
  if (!in_place && (cudaMemcpyAsync(h->st_target, host_target_logits, B * (k + 1) * rowb, H2D, s) != cudaSuccess ||
                    cudaMemcpyAsync(h->st_draft, host_draft_logits, B * k * rowb, H2D, s) != cudaSuccess))
    return SV_ERR_CUDA;
  if (cudaMemcpyAsync(h->st_tokens, host_draft_tokens, B * k * 4, H2D, s) != cudaSuccess ||
      cudaMemcpyAsync(h->st_temp, host_temperature, B * 4, H2D, s) != cudaSuccess ||
      cudaMemcpyAsync(h->st_unif, host_uniforms, B * (k + 1) * 4, H2D, s) != cudaSuccess)
    return SV_ERR_CUDA;
  int rc = verify_impl(h, batch, in_place ? dev_t : h->st_target, in_place ? dev_d : h->st_draft, h->st_tokens,
                       h->st_temp, h->st_unif, h->st_out_tokens, h->st_out_tau,
                       host_out_p_draft ? h->st_out_p : nullptr, host_out_q_draft ? h->st_out_q : nullptr,
                       host_out_tv ? h->st_out_tv : nullptr, nullptr, nullptr, cuda_stream, !in_place);
  if (rc != SV_OK) return rc;
  if (cudaMemcpyAsync(host_out_tokens, h->st_out_tokens, B * (k + 1) * 4, D2H, s) != cudaSuccess ||
      cudaMemcpyAsync(host_out_tau, h->st_out_tau, B * 4, D2H, s) != cudaSuccess)
    return SV_ERR_CUDA;
  if (host_out_p_draft && cudaMemcpyAsync(host_out_p_draft, h->st_out_p, B * k * 4, D2H, s) != cudaSuccess) return SV_ERR_CUDA;
  if (host_out_q_draft && cudaMemcpyAsync(host_out_q_draft, h->st_out_q, B * k * 4, D2H, s) != cudaSuccess) return SV_ERR_CUDA;
  if (host_out_tv && cudaMemcpyAsync(host_out_tv, h->st_out_tv, B * k * 4, D2H, s) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

int spec_verify_get_error(spec_verify_t h, int* invalid_count) {
  if (!h) return SV_ERR_ARG;
  if (invalid_count) *invalid_count = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return SV_ERR_CUDA;
  int f[4] = {0, 0, 0, 0};
  if (cudaMemcpy(f, h->d_flags, sizeof f, cudaMemcpyDeviceToHost) != cudaSuccess) return SV_ERR_CUDA;
  if (cudaMemset(h->d_flags, 0, sizeof f) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return SV_ERR_CUDA;
  if (invalid_count) *invalid_count = f[0];
  if (f[1]) return SV_ERR_TIMEOUT;
  if (f[0]) return SV_ERR_DATA;
  return SV_OK;
}

int spec_verify_selftest_wait(spec_verify_t h, int polls, long long* elapsed_cycles) {
  if (!h || polls < 1) return SV_ERR_ARG;
  long long* d = nullptr;
  if (cudaMalloc(&d, 2 * sizeof(long long)) != cudaSuccess) return SV_ERR_ALLOC;
  sv_wait_selftest_kernel<<<1, 32>>>(h->d_flags, polls, d);
  long long c[2] = {0, 0};
  int rc = cudaGetLastError() == cudaSuccess && cudaMemcpy(c, d, sizeof c, cudaMemcpyDeviceToHost) == cudaSuccess
               ? SV_OK : SV_ERR_CUDA;
  cudaFree(d);
  if (rc != SV_OK) return rc;
  if (elapsed_cycles) {
    elapsed_cycles[0] = c[0];
    elapsed_cycles[1] = c[1];
  }
  int f[2] = {0, 0};   // read without clearing: the flag stays set until spec_verify_get_error
  if (cudaMemcpy(f, h->d_flags, sizeof f, cudaMemcpyDeviceToHost) != cudaSuccess) return SV_ERR_CUDA;
  return f[1] ? SV_ERR_TIMEOUT : f[0] ? SV_ERR_DATA : SV_OK;
}

int spec_verify_info(spec_verify_t h, int* cluster_size, int* n_clusters, int* rounds, int* tma, int* launches_per_call) {
  if (!h) return SV_ERR_ARG;
  if (cluster_size) *cluster_size = h->C;
  if (n_clusters) *n_clusters = h->n_clusters;
  if (rounds) *rounds = h->R;
  if (tma) *tma = h->tma_ok;
  if (launches_per_call) *launches_per_call = 2;   // verification kernel + finalize kernel
  return SV_OK;
}

int spec_verify_kernel_times(spec_verify_t h, float* out_ms, int max_n, int* n_out) {
  if (!h || !h->ev || max_n < 0 || (max_n > 0 && !out_ms)) return SV_ERR_ARG;
  const int n = h->ev_n < max_n ? h->ev_n : max_n;
  for (int i = 0; i < n; ++i) {
    if (cudaEventSynchronize(h->ev[2 * i + 1]) != cudaSuccess) return SV_ERR_CUDA;
    if (cudaEventElapsedTime(&out_ms[i], h->ev[2 * i], h->ev[2 * i + 1]) != cudaSuccess) return SV_ERR_CUDA;
  }
  if (n_out) *n_out = n;
  h->ev_n = 0;
  return SV_OK;
}

void spec_verify_destroy(spec_verify_t h) { free_ctx(h); }

}  // extern "C"
