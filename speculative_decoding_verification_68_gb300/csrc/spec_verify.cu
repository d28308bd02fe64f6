// spec_verify: batched speculative-decoding verification by rejection sampling
// on one GB300 (sm_103a).  The C interface and the method are described in
// include/spec_verify.h; this file holds the kernels and the host side.
//
// Design (one pass over HBM):
//   * A "unit" is one position of one chain: the pair (target row i, draft
//     row i) for i < k, or the single bonus target row k.  Every unit is
//     processed by one thread-block cluster of C CTAs (C <= 8); CTA r owns the
//     vocabulary slice [r*Vs, (r+1)*Vs) of both rows.
//   * The kernel is persistent: each cluster walks units cluster_id,
//     cluster_id + n_clusters, ...  Two CTAs share an SM.  Each CTA has one
//     shared-memory stage; a bulk (TMA) copy lands the next unit's slice there
//     while the current unit is processed from registers.
//   * Pass A (registers): per-row maximum, then sum of exp2(z*c - R) with an
//     integer reference R = ceil(max*c), c = log2(e)/T.  Integer references
//     make every rescale between warps and CTAs an exact power of two.
//   * Exchange 1 (DSMEM push + cluster barrier): per-CTA (max, sum) of both
//     rows; every CTA merges the same values in the same order.
//   * Pass B (registers): with e_j = 2^(z_j*c - R) and r = S_t/S_d, the
//     weight w_j = max(0, e_t - r*e_d) = S_t * max(0, p_j - q_j) (one rounding,
//     exactly zero for identical rows); per-thread, per-round partial sums.
//     The CTA owning the drafted token evaluates the accept test.
//   * Exchange 2: per-CTA residual mass W_c and the accept decision.  The sum
//     of W_c divided by S_t is the TV distance.  If the draft was rejected (or the unit is
//     the bonus row) the CTA whose slice contains u*S draws the token by a
//     hierarchical inverse-CDF search (round/warp table, lane scan, element).
//     The draw is made for every rejected position, so no second pass over
//     HBM is needed once tau is known.
//   * A small finalize kernel (one warp per chain) finds the first rejection
//     with a ballot and writes tokens and tau.
//   Greedy chains (T == 0) use only the maximum and its lowest index.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#include "spec_verify.h"

namespace {

constexpr int NT = 256;            // threads per CTA
constexpr int NWARP = NT / 32;
constexpr int CMAX = 8;            // largest cluster
constexpr int SMALL_BYTES = 6144;  // bookkeeping area in front of the stage
constexpr float LOG2E_F = 1.44269504088896341f;
constexpr float REF_LIMIT = 4194304.0f;   // |max * c| must stay below 2^22
constexpr unsigned FULL = 0xffffffffu;

// status bits of a unit
constexpr int ST_TEMP = 1, ST_TOKEN = 2, ST_ROW = 4;

struct KParams {
  const void* target;        // [B, k+1, V]
  const void* draft;         // [B, k, V]
  const int32_t* tokens;     // [B, k]
  const float* temperature;  // [B]
  const float* uniforms;     // [B, k+1]
  float* out_p;              // [B, k] or null
  float* out_q;              // [B, k] or null
  float* out_tv;             // [B, k] or null
  int32_t* ws_acc;           // [B, k]
  int32_t* ws_y;             // [B, k+1]
  int32_t* ws_status;        // [B, k+1]
  int* flags;                // [0] invalid count, [1] wait timeout
  int B, k, V, Vs;
  int wv;                    // vectors per warp: ceil(ceil(Vs / EPV) / NWARP)
  int units_per_chain;       // k+1 (verify) or k (TV only)
  int tv_only;
  int tma;
};

struct alignas(16) X1 {       // one warp's part of exchange 1 (32 bytes)
  float m_t, m_d;              // maxima of the warp's range in the target / draft row
  float s_t, s_d;              // sums of 2^(z*c - ref(m)) over the range
  int i_t, i_d;                // lowest index of the maximum (T == 0)
  int pad0, pad1;
};
struct alignas(8) X2 {         // one warp's part of exchange 2 (8 bytes)
  float w;                     // residual (or target) weight of the warp's range
  int acc;                     // accept decision if the warp owns the drafted token, else -1
};

struct Small {
  unsigned long long bar;      // stage mbarrier
  int pad0[2];
  X1 x1[2][CMAX * NWARP];      // double-buffered exchange slots, written by peers
  X2 x2[2][CMAX * NWARP];
  float gz_t, gz_d;            // logits at the drafted token (owner CTA)
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

__device__ __forceinline__ void st_peer_x1(uint32_t a, const X1& v) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(__float_as_uint(v.m_t)),
               "r"(__float_as_uint(v.m_d)), "r"(__float_as_uint(v.s_t)), "r"(__float_as_uint(v.s_d)) : "memory");
  asm volatile("st.shared::cluster.v2.b32 [%0], {%1, %2};" ::"r"(a + 16), "r"(v.i_t), "r"(v.i_d) : "memory");
}
__device__ __forceinline__ void st_peer_x2(uint32_t a, const X2& v) {
  asm volatile("st.shared::cluster.v2.b32 [%0], {%1, %2};" ::"r"(a), "r"(__float_as_uint(v.w)), "r"(v.acc) : "memory");
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
__device__ __forceinline__ void mbar_wait_bounded(uint32_t a, unsigned parity, int* flags) {
  for (int it = 0; it < (1 << 22); ++it) {
    if (mbar_try(a, parity)) return;
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
__device__ __forceinline__ int warp_max_s32(int v) { int y; asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(y) : "r"(v)); return y; }
// 2^n for an integer-valued n <= 0, exact (0 below the normal range)
__device__ __forceinline__ float pow2_int(float n) {
  const int e = (int)n;
  return e < -126 ? 0.0f : __int_as_float((e + 127) << 23);
}
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
// integer log2-domain reference for a row maximum m (0 for an empty/invalid part)
__device__ __forceinline__ float ref_of(float m, float c) {
  float r = ceilf(m * c);
  return (isfinite(m) && isfinite(r)) ? r : 0.0f;
}

// ------------------------------------------------------------ per-type access
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

template <typename Tl> __device__ __forceinline__ float vec_max(const uint4& v);
template <> __device__ __forceinline__ float vec_max<float>(const uint4& v) {
  return nanmax(nanmax(__uint_as_float(v.x), __uint_as_float(v.y)), nanmax(__uint_as_float(v.z), __uint_as_float(v.w)));
}
template <> __device__ __forceinline__ float vec_max<__nv_bfloat16>(const uint4& v) {
  __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
  __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
  __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
  __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
  __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
  return nanmax(__low2float(m), __high2float(m));
}

// Sum over one vector of 2^(z*c + nref), as a packed pair accumulator.
template <typename Tl> __device__ __forceinline__ u64 vec_expsum(const uint4& v, u64 cc, u64 nr);
template <> __device__ __forceinline__ u64 vec_expsum<float>(const uint4& v, u64 cc, u64 nr) {
  float a0, a1, a2, a3;
  upk(fma2(pk(__uint_as_float(v.x), __uint_as_float(v.y)), cc, nr), a0, a1);
  upk(fma2(pk(__uint_as_float(v.z), __uint_as_float(v.w)), cc, nr), a2, a3);
  return add2(pk(ex2(a0), ex2(a1)), pk(ex2(a2), ex2(a3)));
}
template <> __device__ __forceinline__ u64 vec_expsum<__nv_bfloat16>(const uint4& v, u64 cc, u64 nr) {
  float a0, a1, a2, a3, a4, a5, a6, a7;
  upk(fma2(pk(bf_lo(v.x), bf_hi(v.x)), cc, nr), a0, a1);
  upk(fma2(pk(bf_lo(v.y), bf_hi(v.y)), cc, nr), a2, a3);
  upk(fma2(pk(bf_lo(v.z), bf_hi(v.z)), cc, nr), a4, a5);
  upk(fma2(pk(bf_lo(v.w), bf_hi(v.w)), cc, nr), a6, a7);
  return add2(add2(pk(ex2(a0), ex2(a1)), pk(ex2(a2), ex2(a3))), add2(pk(ex2(a4), ex2(a5)), pk(ex2(a6), ex2(a7))));
}

// Unscaled residual weights of one pair of elements: max(0, e_t - r * e_d)
// with e = 2^(z*c - R) and r = S_t / S_d, i.e. S_t * max(0, p - q).  One
// rounding after an exact product, so identical rows give exactly zero.
__device__ __forceinline__ u64 pair_w(float t0, float t1, float d0, float d1, u64 cc, u64 nrt, u64 nrd, u64 nr) {
  float at0, at1, ad0, ad1;
  upk(fma2(pk(t0, t1), cc, nrt), at0, at1);
  upk(fma2(pk(d0, d1), cc, nrd), ad0, ad1);
  float w0, w1;
  upk(fma2(pk(ex2(ad0), ex2(ad1)), nr, pk(ex2(at0), ex2(at1))), w0, w1);
  return pk(fmaxf(w0, 0.0f), fmaxf(w1, 0.0f));
}
// Unscaled target weights of one pair of elements: e_t = S_t * p.
__device__ __forceinline__ u64 pair_p(float t0, float t1, u64 cc, u64 nrt) {
  float at0, at1;
  upk(fma2(pk(t0, t1), cc, nrt), at0, at1);
  return pk(ex2(at0), ex2(at1));
}

// Sum of the weights of one vector (residual if PAIR, else target).
template <typename Tl, bool PAIR>
__device__ __forceinline__ float vec_weight_sum(const uint4& t, const uint4& d, u64 cc, u64 nrt, u64 nrd, u64 nr) {
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
__device__ __forceinline__ void vec_weights(const uint4& t, const uint4& d, bool pair, u64 cc, u64 nrt, u64 nrd, u64 nr,
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

// ------------------------------------------------------------- fused kernel
// Vector v of a CTA's slice (16 bytes: EPV logits) belongs to warp v / WV,
// round (v % WV) / 32, lane v % 32, where WV = ceil(nvec / NWARP): every warp
// owns a contiguous range of the vocabulary, and warps are ordered like the
// vocabulary, so (rank, warp) partials are already in index order.
template <typename Tl, int R>
__global__ void __launch_bounds__(NT, 2) sv_fused_kernel(const KParams P) {
  constexpr int EPV = Lay<Tl>::EPV;
  constexpr int ES = (int)sizeof(Tl);
  extern __shared__ __align__(128) unsigned char smem[];
  Small& S = *reinterpret_cast<Small*>(smem);
  float* wsm = reinterpret_cast<float*>(smem + SMALL_BYTES);                 // [R][NT] round weights
  const uint4* stage_t = reinterpret_cast<const uint4*>(smem + SMALL_BYTES + R * NT * 4);
  const uint4* stage_d = reinterpret_cast<const uint4*>(smem + SMALL_BYTES + R * NT * 4 + (size_t)P.Vs * ES);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned C = cl_size(), rank = cl_rank();
  const unsigned cid = cl_id(), ncl = cl_count();
  const int k = P.k, V = P.V, upc = P.units_per_chain;
  const int items = (int)C * NWARP;                     // exchange items per cluster
  const long long slice0 = (long long)rank * P.Vs;
  const int slen = (int)max(0LL, min((long long)P.Vs, (long long)V - slice0));
  const int nvec = (slen + EPV - 1) / EPV;
  const int WV = P.wv;                                  // vectors per warp
  const int vbeg = warp * WV;
  const int vend = min(vbeg + WV, nvec);
  const long long n_units = (long long)P.B * upc;
  const uint32_t bar = saddr(&S.bar);
  const uint32_t stage_t_s = saddr(stage_t), stage_d_s = saddr(stage_d);

  if (tid == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  cluster_sync_all();   // every peer's shared memory is live before the first remote store

  auto unit_rows = [&](long long u, long long& trow, long long& drow, int& ipos, int& b, bool& pair) {
    b = (int)(u / upc);
    ipos = (int)(u % upc);
    pair = ipos < k;
    trow = (long long)b * (k + 1) + ipos;
    drow = (long long)b * k + ipos;
  };
  auto issue_load = [&](long long u) {   // thread 0 only
    long long trow, drow; int ipos, b; bool pair;
    unit_rows(u, trow, drow, ipos, b, pair);
    if (slen > 0) {
      const unsigned bytes = (unsigned)slen * ES;
      mbar_expect_tx(bar, pair ? 2 * bytes : bytes);
      bulk_g2s(stage_t_s, (const char*)P.target + ((size_t)trow * V + slice0) * ES, bytes, bar);
      if (pair) bulk_g2s(stage_d_s, (const char*)P.draft + ((size_t)drow * V + slice0) * ES, bytes, bar);
    } else {
      mbar_arrive(bar);
    }
  };

  long long u = cid;
  if (P.tma && tid == 0 && u < n_units) issue_load(u);
  unsigned phase = 0;
  int n1 = 0, n2 = 0;   // exchanges of each kind performed (select the slot set)

  for (; u < n_units; u += ncl, phase ^= 1u) {
    long long trow, drow; int ipos, b; bool pair;
    unit_rows(u, trow, drow, ipos, b, pair);

    // ---------------- bring this warp's vectors of the unit into registers
    uint4 rt[R], rd[R];
    if (P.tma) {
      mbar_wait_bounded(bar, phase, P.flags);
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int v = vbeg + j * 32 + lane;
        rt[j] = v < vend ? stage_t[v] : Lay<Tl>::neg_inf();
        rd[j] = (pair && v < vend) ? stage_d[v] : Lay<Tl>::neg_inf();
      }
    } else {
      const char* tb = (const char*)P.target + ((size_t)trow * V + slice0) * ES;
      const char* db = (const char*)P.draft + ((size_t)drow * V + slice0) * ES;
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int v = vbeg + j * 32 + lane;
        const bool vin = v < vend;
        uint32_t wt[4], wd[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t xt = 0, xd = 0;
#pragma unroll
          for (int h = 0; h < 4 / ES; ++h) {   // 1 fp32 or 2 bf16 per 32-bit word
            const int e = q * (4 / ES) + h;
            const long long idx = (long long)v * EPV + e;
            const bool in = vin && idx < slen;
            if (ES == 4) {
              xt = in ? ((const uint32_t*)tb)[idx] : 0xff800000u;
              xd = (pair && in) ? ((const uint32_t*)db)[idx] : 0xff800000u;
            } else {
              const uint32_t bt = in ? ((const uint16_t*)tb)[idx] : 0xff80u;
              const uint32_t bd = (pair && in) ? ((const uint16_t*)db)[idx] : 0xff80u;
              xt |= bt << (16 * h); xd |= bd << (16 * h);
            }
          }
          wt[q] = xt; wd[q] = xd;
        }
        rt[j] = make_uint4(wt[0], wt[1], wt[2], wt[3]);
        rd[j] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      }
    }

    // ---------------- per-chain scalars (identical in every CTA of the cluster)
    const float T = P.temperature[b];
    const int x = pair && !P.tv_only ? P.tokens[(size_t)b * k + ipos] : 0;
    const float u_acc = pair && !P.tv_only ? P.uniforms[(size_t)b * (k + 1) + ipos] : 0.0f;
    const float u_fin = P.tv_only ? 0.0f : P.uniforms[(size_t)b * (k + 1) + k];
    const bool t_ok = T >= 0.0f && T <= 3.0e38f;   // false for NaN and inf
    const bool greedy = !(T > 0.0f) || !t_ok;      // invalid temperatures take the cheap path
    const bool x_ok = !pair || P.tv_only || (x >= 0 && x < V);
    const bool own_x = pair && !P.tv_only && x_ok && (long long)x >= slice0 && (long long)x < slice0 + slen;
    if (tid == 0 && own_x) {
      const long long lx = x - slice0;
      if (P.tma) {
        S.gz_t = Lay<Tl>::load_scalar(stage_t, lx);
        S.gz_d = Lay<Tl>::load_scalar(stage_d, lx);
      } else {
        S.gz_t = Lay<Tl>::load_scalar(P.target, (long long)trow * V + x);
        S.gz_d = Lay<Tl>::load_scalar(P.draft, (long long)drow * V + x);
      }
    }
    __syncthreads();   // stage fully consumed; gathered values visible
    if (P.tma && tid == 0 && u + ncl < n_units) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue_load(u + ncl);
    }

    const float c = greedy ? 0.0f : fminf(__fdiv_rn(LOG2E_F, T), 3.0e38f);

    // ---------------- pass A: per-warp statistics, pushed to every CTA of the cluster
    float tm_t = -INFINITY, tm_d = -INFINITY;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      tm_t = nanmax(tm_t, vec_max<Tl>(rt[j]));
      if (pair) tm_d = nanmax(tm_d, vec_max<Tl>(rd[j]));
    }
    X1 mine;
    mine.m_t = warp_max_nan(tm_t);
    mine.m_d = pair ? warp_max_nan(tm_d) : -INFINITY;
    mine.i_t = 0x7fffffff; mine.i_d = 0x7fffffff;
    mine.s_t = 0.0f; mine.s_d = 0.0f;
    if (greedy) {
      int ci_t = 0x7fffffff, ci_d = 0x7fffffff;   // lowest global index holding the warp maximum
#pragma unroll
      for (int j = R - 1; j >= 0; --j) {
#pragma unroll
        for (int e = EPV - 1; e >= 0; --e) {
          const int gi = (int)slice0 + (vbeg + j * 32 + lane) * EPV + e;
          if (Lay<Tl>::elem(rt[j], e) == mine.m_t) ci_t = gi;
          if (pair && Lay<Tl>::elem(rd[j], e) == mine.m_d) ci_d = gi;
        }
      }
      mine.i_t = (int)warp_min_u32((unsigned)ci_t);
      mine.i_d = (int)warp_min_u32((unsigned)ci_d);
    } else {
      const u64 cc = pk(c, c);
      const float rwt = ref_of(mine.m_t, c), rwd = ref_of(mine.m_d, c);
      const u64 nrt = pk(-rwt, -rwt), nrd = pk(-rwd, -rwd);
      u64 at = 0ull, ad = 0ull;
#pragma unroll
      for (int j = 0; j < R; ++j) {
        at = add2(at, vec_expsum<Tl>(rt[j], cc, nrt));
        if (pair) ad = add2(ad, vec_expsum<Tl>(rd[j], cc, nrd));
      }
      float lo, hi;
      upk(at, lo, hi);
      mine.s_t = warp_sum_f32(lo + hi);
      upk(ad, lo, hi);
      mine.s_d = pair ? warp_sum_f32(lo + hi) : 0.0f;
    }
    const int set1 = n1 & 1;
    if (lane < (int)C) st_peer_x1(peer_addr(saddr(&S.x1[set1][rank * NWARP + warp]), lane), mine);
    cluster_sync_all();
    ++n1;

    // Cluster merge, identical in every warp: lane l holds items l and l + 32.
    X1 ia, ib;
    {
      X1 z;
      z.m_t = -INFINITY; z.m_d = -INFINITY; z.s_t = 0.0f; z.s_d = 0.0f; z.i_t = 0x7fffffff; z.i_d = 0x7fffffff;
      ia = lane < items ? S.x1[set1][lane] : z;
      ib = lane + 32 < items ? S.x1[set1][lane + 32] : z;
    }
    const float M_t = warp_max_nan(nanmax(ia.m_t, ib.m_t));
    const float M_d = warp_max_nan(nanmax(ia.m_d, ib.m_d));
    int A_t = 0, A_d = 0;
    float S_t = 0.0f, S_d = 0.0f;
    float pa = 0.0f, pb = 0.0f;   // items' shares of sum_j e_t (fallback draw)
    float R_t = 0.0f, R_d = 0.0f;
    if (greedy) {
      A_t = (int)warp_min_u32((unsigned)min(ia.m_t == M_t ? ia.i_t : 0x7fffffff, ib.m_t == M_t ? ib.i_t : 0x7fffffff));
      A_d = (int)warp_min_u32((unsigned)min(ia.m_d == M_d ? ia.i_d : 0x7fffffff, ib.m_d == M_d ? ib.i_d : 0x7fffffff));
    } else {
      R_t = ref_of(M_t, c);
      R_d = ref_of(M_d, c);
      pa = ia.s_t * pow2_int(ref_of(ia.m_t, c) - R_t);
      pb = ib.s_t * pow2_int(ref_of(ib.m_t, c) - R_t);
      S_t = warp_sum_f32(pa + pb);
      S_d = warp_sum_f32(ia.s_d * pow2_int(ref_of(ia.m_d, c) - R_d) + ib.s_d * pow2_int(ref_of(ib.m_d, c) - R_d));
    }
    bool row_ok = isfinite(M_t) && (!pair || isfinite(M_d));
    if (!greedy) {
      row_ok = row_ok && fabsf(M_t * c) < REF_LIMIT && S_t > 0.0f && isfinite(S_t);
      if (pair) row_ok = row_ok && fabsf(M_d * c) < REF_LIMIT && S_d > 0.0f && isfinite(S_d);
    }
    const int status = (t_ok ? 0 : ST_TEMP) | (x_ok ? 0 : ST_TOKEN) | (row_ok ? 0 : ST_ROW);
    const size_t ui = (size_t)b * (k + 1) + ipos;   // unit index within [B, k+1]
    const size_t pi = (size_t)b * k + ipos;         // position index within [B, k]

    if (status != 0 || greedy) {
      if (rank == 0 && tid == 0) {
        if (!P.tv_only) {
          P.ws_status[ui] = status;
          if (status == 0) {
            P.ws_y[ui] = A_t;
            if (pair) {
              P.ws_acc[pi] = x == A_t;
              if (P.out_p) P.out_p[pi] = x == A_t ? 1.0f : 0.0f;
              if (P.out_q) P.out_q[pi] = x == A_d ? 1.0f : 0.0f;
            }
          }
        } else if (status != 0) {
          atomicAdd(&P.flags[0], 1);
        }
        if (pair && P.out_tv) P.out_tv[pi] = status == 0 ? (A_t != A_d ? 1.0f : 0.0f) : __int_as_float(0x7fc00000);
      }
      continue;   // cluster-uniform: every CTA took the same branch
    }

    // ---------------- pass B: residual (pair) or target (bonus) weights, unscaled
    const u64 cc = pk(c, c);
    const u64 nrt = pk(-R_t, -R_t), nrd = pk(-R_d, -R_d);
    const float r_f = pair ? S_t / S_d : 0.0f;   // q_j = e_d * r / S_t
    const u64 nr = pk(-r_f, -r_f);
    float wthr = 0.0f;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const float wj = pair ? vec_weight_sum<Tl, true>(rt[j], rd[j], cc, nrt, nrd, nr)
                            : vec_weight_sum<Tl, false>(rt[j], rd[j], cc, nrt, nrd, nr);
      wsm[j * NT + tid] = wj;
      wthr += wj;
    }
    X2 mine2;
    mine2.w = warp_sum_f32(wthr);
    mine2.acc = -1;
    if (own_x && tid == 0) {   // accept test at the drafted token (owner CTA, one thread)
      const float lpx = fmaf(S.gz_t, c, -R_t), lqx = fmaf(S.gz_d, c, -R_d);
      const float ratio = exp2f(lpx - lqx) * (S_d / S_t);
      mine2.acc = u_acc < ratio ? 1 : 0;
      P.ws_acc[pi] = mine2.acc;
      if (P.out_p) P.out_p[pi] = exp2f(lpx) / S_t;
      if (P.out_q) P.out_q[pi] = exp2f(lqx) / S_d;
    }
    mine2.acc = __shfl_sync(FULL, mine2.acc, 0);

    // ---------------- exchange 2: per-warp residual mass and the accept decision
    const int set2 = n2 & 1;
    if (lane < (int)C) st_peer_x2(peer_addr(saddr(&S.x2[set2][rank * NWARP + warp]), lane), mine2);
    cluster_sync_all();
    ++n2;

    // lane l holds items 2l and 2l+1 (vocabulary order)
    X2 ja, jb;
    ja.w = 0.0f; ja.acc = -1; jb.w = 0.0f; jb.acc = -1;
    if (2 * lane < items) ja = S.x2[set2][2 * lane];
    if (2 * lane + 1 < items) jb = S.x2[set2][2 * lane + 1];
    const int acc_all = warp_max_s32(max(ja.acc, jb.acc));
    const float res_total = warp_sum_f32(ja.w + jb.w);                    // S_t * TV
    const bool fallback = pair && !(res_total > 0.0f);                     // zero residual: draw from p
    double wa = ja.w, wb = jb.w;
    if (fallback) {   // the p shares of items 2l, 2l+1 live in lanes l and l+16 (as items l, l+32)
      const int ka = 2 * lane, kb = 2 * lane + 1;
      const float a0 = __shfl_sync(FULL, pa, ka & 31), a1 = __shfl_sync(FULL, pb, ka & 31);
      const float b0 = __shfl_sync(FULL, pa, kb & 31), b1 = __shfl_sync(FULL, pb, kb & 31);
      wa = ka < items ? (ka < 32 ? a0 : a1) : 0.0f;
      wb = kb < items ? (kb < 32 ? b0 : b1) : 0.0f;
    }
    double incl = wa + wb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += y;
    }
    double excl = __shfl_up_sync(FULL, incl, 1);
    if (lane == 0) excl = 0.0;
    const double total = __shfl_sync(FULL, incl, 31);

    if (rank == 0 && tid == 0) {
      if (pair && P.out_tv) P.out_tv[pi] = res_total / S_t;
      if (!P.tv_only) P.ws_status[ui] = 0;
    }
    if (P.tv_only || (pair && acc_all == 1)) continue;   // no draw needed for this unit

    // ---------------- inverse-CDF draw: which (CTA, warp) holds u * total
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
    if (item != (int)rank * NWARP + warp) continue;   // only the owning warp draws

    // Owner warp: round totals, then the lane, then the element.
    const bool use_pair = pair && !fallback;
    float wl[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
      wl[j] = fallback ? vec_weight_sum<Tl, false>(rt[j], rd[j], cc, nrt, nrd, nr) : wsm[j * NT + tid];
    }
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
    if (jstar < 0) continue;   // nothing positive (cannot happen for a valid owner)
    float mw = 0.0f;
#pragma unroll
    for (int j = 0; j < R; ++j) if (j == jstar) mw = wl[j];
    double inc = (double)mw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(FULL, inc, o);
      if (lane >= o) inc += y;
    }
    const unsigned h2 = __ballot_sync(FULL, !over && mw > 0.0f && tin < inc);
    const unsigned p2 = __ballot_sync(FULL, mw > 0.0f);
    int lstar;
    if (h2) lstar = __ffs(h2) - 1;
    else { lstar = 31 - __clz(p2); over = true; }
    const double t2 = tin - (__shfl_sync(FULL, inc, lstar) - (double)__shfl_sync(FULL, mw, lstar));
    if (lane == lstar) {
      float w[EPV];
#pragma unroll
      for (int e = 0; e < EPV; ++e) w[e] = 0.0f;
#pragma unroll
      for (int j = 0; j < R; ++j)
        if (j == jstar) vec_weights<Tl>(rt[j], rd[j], use_pair, cc, nrt, nrd, nr, w);
      int estar = -1, elast = 0;
      double run2 = 0.0;
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        if (w[e] > 0.0f) elast = e;
        if (!over && estar < 0 && w[e] > 0.0f && t2 < run2 + (double)w[e]) estar = e;
        run2 += (double)w[e];
      }
      if (estar < 0) estar = elast;
      P.ws_y[ui] = (int)slice0 + (vbeg + jstar * 32 + lstar) * EPV + estar;
    }
  }
  cluster_sync_all();   // no CTA leaves while a peer could still address its shared memory
}

// ------------------------------------------------------------ finalize kernel
struct FParams {
  const int32_t* tokens;
  const int32_t* ws_acc;
  const int32_t* ws_y;
  const int32_t* ws_status;
  int32_t* out_tokens;
  int32_t* out_tau;
  int* flags;
  int B, k;
};

__global__ void __launch_bounds__(256) sv_finalize_kernel(const FParams F) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (b >= F.B) return;
  const int k = F.k;
  const int st = lane <= k ? F.ws_status[(size_t)b * (k + 1) + lane] : 0;
  const bool bad = __any_sync(FULL, st != 0);
  const int a = lane < k ? F.ws_acc[(size_t)b * k + lane] : 1;
  const unsigned rej = __ballot_sync(FULL, lane < k && a == 0);
  const int tau = rej ? __ffs(rej) - 1 : k;
  if (bad) {
    if (lane <= k) F.out_tokens[(size_t)b * (k + 1) + lane] = -1;
    if (lane == 0) { F.out_tau[b] = -1; atomicAdd(&F.flags[0], 1); }
    return;
  }
  if (lane <= k) {
    int tok = -1;
    if (lane < tau) tok = F.tokens[(size_t)b * k + lane];
    else if (lane == tau) tok = F.ws_y[(size_t)b * (k + 1) + tau];
    F.out_tokens[(size_t)b * (k + 1) + lane] = tok;
  }
  if (lane == 0) F.out_tau[b] = tau;
}

typedef void (*FusedFn)(const KParams);
constexpr int R_CHOICES[] = {1, 2, 4, 6, 8, 10};
constexpr int N_R = 6;

template <typename Tl>
FusedFn pick_kernel(int r) {
  switch (r) {
    case 1: return sv_fused_kernel<Tl, 1>;
    case 2: return sv_fused_kernel<Tl, 2>;
    case 4: return sv_fused_kernel<Tl, 4>;
    case 6: return sv_fused_kernel<Tl, 6>;
    case 8: return sv_fused_kernel<Tl, 8>;
    default: return sv_fused_kernel<Tl, 10>;
  }
}

}  // namespace

// ------------------------------------------------------------------ host side
struct spec_verify_ctx {
  int device;
  int max_batch, k, V, dtype;
  unsigned flags;
  int C, Vs, R, wv, n_clusters, tma_ok;
  size_t smem;
  FusedFn kernel;
  int32_t* ws_acc;
  int32_t* ws_y;
  int32_t* ws_status;
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

static void free_ctx(spec_verify_ctx* h) {
  if (!h) return;
  void* ptrs[] = {h->ws_acc, h->ws_y, h->ws_status, h->d_flags, h->st_target, h->st_draft, h->st_tokens, h->st_temp,
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

static int launch_fused(spec_verify_ctx* h, const KParams& P, long long units, cudaStream_t s) {
  const int grid_clusters = (int)(units < h->n_clusters ? units : h->n_clusters);
  if (grid_clusters <= 0) return SV_OK;
  const bool timed = h->ev && h->ev_n < TIMING_RING;
  if (timed && cudaEventRecord(h->ev[2 * h->ev_n], s) != cudaSuccess) return SV_ERR_CUDA;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)(grid_clusters * h->C), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = h->smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)h->C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, h->kernel, P) != cudaSuccess) return SV_ERR_CUDA;
  if (timed) {
    if (cudaEventRecord(h->ev[2 * h->ev_n + 1], s) != cudaSuccess) return SV_ERR_CUDA;
    h->ev_n++;
  }
  return SV_OK;
}

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
  const long long wv = (nvec + NWARP - 1) / NWARP;
  const long long r_need = (wv + 31) / 32;
  int R = -1;
  for (int i = 0; i < N_R; ++i)
    if (R_CHOICES[i] >= r_need) { R = R_CHOICES[i]; break; }
  if (R < 0) return SV_ERR_SIZE;

  spec_verify_ctx* h = (spec_verify_ctx*)calloc(1, sizeof(spec_verify_ctx));
  if (!h) return SV_ERR_ALLOC;
  if (cudaGetDevice(&h->device) != cudaSuccess) { free(h); return SV_ERR_CUDA; }
  h->max_batch = max_batch; h->k = k; h->V = vocab; h->dtype = logit_dtype; h->flags = flags;
  h->C = C; h->Vs = (int)Vs; h->R = R; h->wv = (int)wv;
  h->tma_ok = ((size_t)vocab * es) % 16 == 0 && !(flags & SV_FLAG_NO_TMA);
  h->smem = SMALL_BYTES + (size_t)R * NT * 4 + 2 * (size_t)Vs * es;
  h->kernel = logit_dtype == SV_FP32 ? pick_kernel<float>(R) : pick_kernel<__nv_bfloat16>(R);
  if (cudaFuncSetAttribute(h->kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h->smem) != cudaSuccess) {
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
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, h->kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      free_ctx(h);
      return SV_ERR_CUDA;
    }
    h->n_clusters = n;
  }
  const size_t mb = (size_t)(max_batch > 0 ? max_batch : 1);
  bool ok = cudaMalloc(&h->ws_acc, mb * k * sizeof(int32_t)) == cudaSuccess &&
            cudaMalloc(&h->ws_y, mb * (k + 1) * sizeof(int32_t)) == cudaSuccess &&
            cudaMalloc(&h->ws_status, mb * (k + 1) * sizeof(int32_t)) == cudaSuccess &&
            cudaMalloc(&h->d_flags, 4 * sizeof(int)) == cudaSuccess;
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
  if (!h || batch < 0 || batch > h->max_batch) return SV_ERR_ARG;
  if (batch == 0) return SV_OK;
  if (!target_logits || !draft_logits || !draft_tokens || !temperature || !uniforms || !out_tokens || !out_tau)
    return SV_ERR_ARG;
  const int es = h->dtype == SV_FP32 ? 4 : 2;
  if (((uintptr_t)target_logits % es) || ((uintptr_t)draft_logits % es)) return SV_ERR_ARG;
  if (!al4(draft_tokens) || !al4(temperature) || !al4(uniforms) || !al4(out_tokens) || !al4(out_tau) ||
      !al4(out_p_draft) || !al4(out_q_draft) || !al4(out_tv))
    return SV_ERR_ARG;
  cudaStream_t s = (cudaStream_t)cuda_stream;
  KParams P;
  memset(&P, 0, sizeof P);
  P.target = target_logits; P.draft = draft_logits; P.tokens = draft_tokens; P.temperature = temperature;
  P.uniforms = uniforms; P.out_p = out_p_draft; P.out_q = out_q_draft; P.out_tv = out_tv;
  P.ws_acc = h->ws_acc; P.ws_y = h->ws_y; P.ws_status = h->ws_status; P.flags = h->d_flags;
  P.B = batch; P.k = h->k; P.V = h->V; P.Vs = h->Vs; P.wv = h->wv;
  P.units_per_chain = h->k + 1; P.tv_only = 0;
  P.tma = h->tma_ok && al16(target_logits) && al16(draft_logits);
  int rc = launch_fused(h, P, (long long)batch * (h->k + 1), s);
  if (rc != SV_OK) return rc;
  FParams F;
  F.tokens = draft_tokens; F.ws_acc = h->ws_acc; F.ws_y = h->ws_y; F.ws_status = h->ws_status;
  F.out_tokens = out_tokens; F.out_tau = out_tau; F.flags = h->d_flags; F.B = batch; F.k = h->k;
  sv_finalize_kernel<<<(batch + 7) / 8, 256, 0, s>>>(F);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
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
  P.ws_acc = h->ws_acc; P.ws_y = h->ws_y; P.ws_status = h->ws_status; P.flags = h->d_flags;
  P.B = batch; P.k = h->k; P.V = h->V; P.Vs = h->Vs; P.wv = h->wv;
  P.units_per_chain = h->k; P.tv_only = 1;
  P.tma = h->tma_ok && al16(target_logits) && al16(draft_logits);
  return launch_fused(h, P, (long long)batch * h->k, (cudaStream_t)cuda_stream);
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
  if (cudaMemcpyAsync(h->st_target, host_target_logits, B * (k + 1) * rowb, H2D, s) != cudaSuccess ||
      cudaMemcpyAsync(h->st_draft, host_draft_logits, B * k * rowb, H2D, s) != cudaSuccess ||
      cudaMemcpyAsync(h->st_tokens, host_draft_tokens, B * k * 4, H2D, s) != cudaSuccess ||
      cudaMemcpyAsync(h->st_temp, host_temperature, B * 4, H2D, s) != cudaSuccess ||
      cudaMemcpyAsync(h->st_unif, host_uniforms, B * (k + 1) * 4, H2D, s) != cudaSuccess)
    return SV_ERR_CUDA;
  int rc = spec_verify(h, batch, h->st_target, h->st_draft, h->st_tokens, h->st_temp, h->st_unif, h->st_out_tokens,
                       h->st_out_tau, host_out_p_draft ? h->st_out_p : nullptr, host_out_q_draft ? h->st_out_q : nullptr,
                       host_out_tv ? h->st_out_tv : nullptr, cuda_stream);
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

int spec_verify_info(spec_verify_t h, int* cluster_size, int* n_clusters, int* rounds, int* tma, int* launches_per_call) {
  if (!h) return SV_ERR_ARG;
  if (cluster_size) *cluster_size = h->C;
  if (n_clusters) *n_clusters = h->n_clusters;
  if (rounds) *rounds = h->R;
  if (tma) *tma = h->tma_ok;
  if (launches_per_call) *launches_per_call = 2;
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
