// vpd_stream.cu -- streaming kernels: each CTA owns one token row at a time
// (grid-stride over rows) and sweeps the row's vocabulary with coalesced
// 16-byte vector loads, reducing per-thread partials with warp shuffles and
// shared memory.
//
// Sources (web pages):
//   [JSD page] DeepSpeed pull request #8958, "[VocabTP] Add vocabulary-parallel
//              generalized JSD with Triton kernels".
//   [ops page] DeepSpeed pull request #8791, "Add vocabulary-parallel logprobs,
//              entropy and KL ops".
//
// Kernels:
//   k_pair_stats   paired statistics of student and teacher, merged over the
//                  ordered vocabulary segments ([JSD page], "Changes").
//   k_jsd_div      the two KL-to-mixture expectations reduced together; the
//                  second of the two input passes ([JSD page], "Scope and
//                  limitations"); beta = 0 / 1 are explicit KL branches.
//   k_pair_bwd     closed-form backward recomputing P_s, P_t and M in registers
//                  ([JSD page], "Changes"; [ops page], "How").
//   k_kl_fwd       single online pass for KL ([JSD page], "Scope and limitations"
//                  mentions the existing single-pass KL forward).
//   k_entropy_*    entropy forward (one online pass) and backward.
//   k_logprobs_*   selected / top-k log-probabilities and their backward.

#include <cuda_runtime.h>

#include <atomic>
#include <type_traits>

#include "vpd_internal.h"
#include "vpd_packed.cuh"

namespace vpd {
namespace {

constexpr int kUnroll = 4;  // 16-byte vectors per input in flight per thread

// 16-bit inputs can be handed to a body as raw 16-byte vectors (Body::kRaw),
// which it consumes with packed arithmetic instead of unpacked floats.
template <class T>
struct Packed {
  using type = void;
};
template <>
struct Packed<BF16> {
  using type = InBF16;
};
template <>
struct Packed<F16> {
  using type = InF16;
};
template <class B, class = void>
struct HasRaw : std::false_type {};
template <class B>
struct HasRaw<B, std::void_t<decltype(B::kRaw)>> : std::bool_constant<B::kRaw> {};
template <class T, class Body>
constexpr bool kUseRaw = T::kSize == 2 && HasRaw<Body>::value;

// ---------------------------------------------------------------------------
// Row sweeps. The range [0, n) of one row (or of a row pair with the same
// 16-byte phase) is visited as a scalar head up to the first 16-byte boundary,
// a body of whole vectors, and a scalar tail. A row pair whose inputs have
// different 16-byte phases is visited element by element.
// ---------------------------------------------------------------------------
template <class T, class Body>
__device__ __forceinline__ void visit2(const char* a, const char* b, int64_t n, Body& body) {
  constexpr int V = T::kVec;
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  int64_t head = n;
  if (((pa ^ pb) & 15u) == 0) {
    head = static_cast<int64_t>((16u - (pa & 15u)) & 15u) / T::kSize;
    if (head > n) head = n;
  }
  const int64_t tid = threadIdx.x, nt = blockDim.x;
  for (int64_t j = tid; j < head; j += nt) body.one(j, T::load(a, j), T::load(b, j));
  const int64_t nv = (n - head) / V;
  const char* va = a + head * T::kSize;
  const char* vb = b + head * T::kSize;
  int64_t i = tid;
  for (; i + (kUnroll - 1) * nt < nv; i += kUnroll * nt) {
    uint4 ra[kUnroll], rb[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      ra[u] = ldg16(va + (i + u * nt) * 16);
      rb[u] = ldg16(vb + (i + u * nt) * 16);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if constexpr (kUseRaw<T, Body>) {
        body.template raw<typename Packed<T>::type>(head + (i + u * nt) * V, ra[u], rb[u]);
      } else {
        float xa[V], xb[V];
        T::unpack(ra[u], xa);
        T::unpack(rb[u], xb);
        body.vec(head + (i + u * nt) * V, xa, xb);
      }
    }
  }
  for (; i < nv; i += nt) {
    if constexpr (kUseRaw<T, Body>) {
      body.template raw<typename Packed<T>::type>(head + i * V, ldg16(va + i * 16), ldg16(vb + i * 16));
    } else {
      float xa[V], xb[V];
      T::unpack(ldg16(va + i * 16), xa);
      T::unpack(ldg16(vb + i * 16), xb);
      body.vec(head + i * V, xa, xb);
    }
  }
  for (int64_t j = head + nv * V + tid; j < n; j += nt) body.one(j, T::load(a, j), T::load(b, j));
}

// (tid, nt): this thread's place among the nt threads that share the row (the
// CTA, or one warp in the warp-per-row kernels).
template <class T, class Body>
__device__ __forceinline__ void visit1(const char* a, int64_t n, Body& body, int64_t tid = threadIdx.x,
                                       int64_t nt = blockDim.x) {
  constexpr int V = T::kVec;
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a);
  int64_t head = static_cast<int64_t>((16u - (pa & 15u)) & 15u) / T::kSize;
  if (head > n) head = n;
  for (int64_t j = tid; j < head; j += nt) body.one(j, T::load(a, j));
  const int64_t nv = (n - head) / V;
  const char* va = a + head * T::kSize;
  int64_t i = tid;
  for (; i + (kUnroll - 1) * nt < nv; i += kUnroll * nt) {
    uint4 ra[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) ra[u] = ldg16(va + (i + u * nt) * 16);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if constexpr (kUseRaw<T, Body>) {
        body.template raw<typename Packed<T>::type>(head + (i + u * nt) * V, ra[u]);
      } else {
        float xa[V];
        T::unpack(ra[u], xa);
        body.vec(head + (i + u * nt) * V, xa);
      }
    }
  }
  for (; i < nv; i += nt) {
    if constexpr (kUseRaw<T, Body>) {
      body.template raw<typename Packed<T>::type>(head + i * V, ldg16(va + i * 16));
    } else {
      float xa[V];
      T::unpack(ldg16(va + i * 16), xa);
      body.vec(head + i * V, xa);
    }
  }
  for (int64_t j = head + nv * V + tid; j < n; j += nt) body.one(j, T::load(a, j));
}

template <class T>
__device__ __forceinline__ const char* row_ptr(const View& v, int64_t r) {
  return v.data + v.map.offset(r) * T::kSize;
}

// Is p + j elements of size S aligned for an N-element vector store?
template <int S, int N>
__device__ __forceinline__ bool store_aligned(const char* p, int64_t j) {
  constexpr int kBytes = S * N < 16 ? S * N : 16;
  return (reinterpret_cast<uintptr_t>(p + j * S) & (kBytes - 1)) == 0;
}

// Zero a gradient row of n elements.
template <class G>
__device__ void zero_row(char* p, int64_t n) {
  const int64_t tid = threadIdx.x, nt = blockDim.x;
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  int64_t head = static_cast<int64_t>((16u - (a & 15u)) & 15u) / G::kSize;
  if (head > n) head = n;
  for (int64_t j = tid; j < head; j += nt) G::store(p, j, 0.f);
  constexpr int kPer = 16 / G::kSize;
  const int64_t nv = (n - head) / kPer;
  uint4* pv = reinterpret_cast<uint4*>(p + head * G::kSize);
  for (int64_t i = tid; i < nv; i += nt) pv[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t j = head + nv * kPer + tid; j < n; j += nt) G::store(p, j, 0.f);
}

// Per-row statistics as stored in `saved`.
struct RowStat {
  float m;  // max over the support, -inf if empty, NaN if NaN/+inf present
  float L;  // ln of the sum-exp relative to m
};

__device__ __forceinline__ RowStat finish_stat(Stat st) {
  if (stat_bad(st)) return {qnan(), qnan()};
  if (st.m == neg_inf()) return {neg_inf(), neg_inf()};
  return {st.m, logf(st.z)};
}

__device__ __forceinline__ bool stat_ok(RowStat r) { return isfinite(r.m); }

// Online statistics of one raw vector of 8 packed 16-bit values. First the
// running max: the NaN-propagating packed max of the vector (a NaN makes z NaN
// for good); when it grows, `grow(old_m, new_m)` rescales whatever the body
// keeps relative to it, then m moves. Then the exponentials relative to the
// running max with x - m exact: d[w] = (x - m) log2 e and e[w] = 2^d[w] for
// the four packed pairs, and z += sum e. With CLAMP, -inf entries enter as the
// finite floor (e = 0 still, d finite), for bodies that multiply e by d.
template <class In, bool CLAMP, class Grow>
__device__ __forceinline__ void stat_raw(Stat& st, const uint4& v, float2 (&d)[4], float2 (&e)[4], Grow&& grow) {
  const uint32_t mx = In::max_nan(In::max_nan(v.x, v.y), In::max_nan(v.z, v.w));
  const float2 m2 = In::unpack(mx);
  const float vm = max_nan(m2.x, m2.y);
  if (isnan(vm)) {
    st.z = qnan();
  } else if (vm > st.m) {
    grow(st.m, vm);
    if (st.m != neg_inf()) st.z *= exp_acc(st.m - vm);
    st.m = vm;
  }
  const float2 nr2 = f2(-stat_ref(st.m)), l2e2 = f2(kLog2e);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float2 z2 = f2(0.f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    d[i] = mul2(In::sub(CLAMP ? In::max2(w[i], In::kNegBig2) : w[i], nr2), l2e2);
    e[i] = ex2_2(d[i]);
    z2 = add2(z2, e[i]);
  }
  st.z += z2.x + z2.y;
}
struct NoGrow {
  __device__ __forceinline__ void operator()(float, float) const {}
};

// ===========================================================================
// Paired statistics (first input pass of the JSD forward).
// ===========================================================================
struct PairStatBody {
  static constexpr bool kRaw = true;
  Stat s, t;
  template <class In>
  __device__ __forceinline__ void raw(int64_t, const uint4& a, const uint4& b) {
    float2 d[4], e[4];
    stat_raw<In, false>(s, a, d, e, NoGrow{});
    stat_raw<In, false>(t, b, d, e, NoGrow{});
  }
  template <int N>
  __device__ __forceinline__ void vec(int64_t, const float (&xs)[N], const float (&xt)[N]) {
    stat_add<N>(s, xs);
    stat_add<N>(t, xt);
  }
  __device__ __forceinline__ void one(int64_t, float xs, float xt) {
    stat_add1(s, xs);
    stat_add1(t, xt);
  }
};

template <class T>
__global__ void __maxnreg__(56) k_pair_stats(View s, View t, Segs seg, float* saved) {
  __shared__ float scratch[2 * 64];
  for (int64_t r = blockIdx.x; r < s.rows; r += gridDim.x) {
    const char* ps = row_ptr<T>(s, r);
    const char* pt = row_ptr<T>(t, r);
    Stat run[2] = {stat_init(), stat_init()};
    for (int k = 0; k < seg.count; ++k) {
      const int64_t off = seg.off[k], w = seg.off[k + 1] - off;
      PairStatBody b{stat_init(), stat_init()};
      visit2<T>(ps + off * T::kSize, pt + off * T::kSize, w, b);
      Stat part[2] = {b.s, b.t};
      block_stat<2>(part, scratch);
      // segment merge in segment order: MAX of maxima, SUM of rescaled sums
      run[0] = stat_merge(run[0], part[0]);
      run[1] = stat_merge(run[1], part[1]);
    }
    if (threadIdx.x == 0) {
      RowStat a = finish_stat(run[0]), c = finish_stat(run[1]);
      float* o = saved + r * VPD_SAVED_PAIR;
      o[0] = a.m;
      o[1] = a.L;
      o[2] = c.m;
      o[3] = c.L;
    }
  }
}

// ===========================================================================
// Per-element JSD quantities from the two log-probabilities.
// lp, lq are ln p_j, ln q_j (-inf on masked tokens; not both -inf when used).
// Returns p, q and ln M_j = ln((1-beta) p_j + beta q_j), evaluated as
// hi + ln(w_hi + w_lo e^{lo - hi}) so no underflow reaches the logarithm.
// ===========================================================================
struct Mix {
  float ws, wt;  // 1 - beta, beta
};

__device__ __forceinline__ void mix_terms(float lp, float lq, const Mix& c, float& p, float& q,
                                          float& lm) {
  const bool p_hi = lp >= lq;
  const float hi = p_hi ? lp : lq;
  const float lo = p_hi ? lq : lp;
  const float r = expd(lo - hi);
  const float e = expd(hi);
  const float w_hi = p_hi ? c.ws : c.wt;
  const float w_lo = p_hi ? c.wt : c.ws;
  lm = hi + kLn2 * lg2(fmaf(w_lo, r, w_hi));
  p = p_hi ? e : e * r;
  q = p_hi ? e * r : e;
}

enum Mode : int { kInterior = 0, kForwardKL = 1, kReverseKL = 2 };

// Raw 16-bit vectors of a row pair with known statistics, in log2 units:
// log2 p = (s - m_s) log2 e - L_s log2 e (x - m exact), p = 2^log2 p, and the
// same for q. -inf logits enter as the finite floor, so their p or q is 0 and
// every product with a log-ratio stays finite.
constexpr float kTinyMix = 1e-37f;  // keeps M > 0 so log2 M stays finite
template <class In>
__device__ __forceinline__ void pair_log2(uint32_t ws, uint32_t wt, float2 nms2, float2 nmt2, float2 nKs2,
                                          float2 nKt2, float2& lp, float2& lq, float2& p, float2& q) {
  const float2 l2e2 = f2(kLog2e);
  lp = fma2(In::sub(In::max2(ws, In::kNegBig2), nms2), l2e2, nKs2);
  lq = fma2(In::sub(In::max2(wt, In::kNegBig2), nmt2), l2e2, nKt2);
  p = ex2_2(lp);
  q = ex2_2(lq);
}

// ===========================================================================
// Divergence pass (second input pass of the JSD forward).
// ===========================================================================
template <int MODE>
struct DivBody {
  static constexpr bool kRaw = true;
  float ms, Ls, mt, Lt;
  Mix mix;
  float A, B;  // interior: the two KL-to-mixture sums; endpoints: A holds the KL sum
  int viol;    // endpoints: the target has a finite logit where the other is -inf

  template <class In>
  __device__ __forceinline__ void raw(int64_t, const uint4& a, const uint4& b) {
    const float2 nms2 = f2(-ms), nmt2 = f2(-mt), nKs2 = f2(-Ls * kLog2e), nKt2 = f2(-Lt * kLog2e);
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
    float2 acc_a = f2(0.f), acc_b = f2(0.f);
    uint32_t v = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 lp, lq, p, q;
      pair_log2<In>(wa[i], wb[i], nms2, nmt2, nKs2, nKt2, lp, lq, p, q);
      if (MODE == kInterior) {
        const float2 lm = lg2_2(fma2(f2(mix.ws), p, fma2(f2(mix.wt), q, f2(kTinyMix))));
        acc_a = fma2(q, add2(lq, neg(lm)), acc_a);
        acc_b = fma2(p, add2(lp, neg(lm)), acc_b);
      } else if (MODE == kForwardKL) {  // KL(q || p)
        acc_a = fma2(q, add2(lq, neg(lp)), acc_a);
        v |= __vcmpeq2(wa[i], In::kNegInf2) & ~__vcmpeq2(wb[i], In::kNegInf2);
      } else {  // KL(p || q)
        acc_a = fma2(p, add2(lp, neg(lq)), acc_a);
        v |= __vcmpeq2(wb[i], In::kNegInf2) & ~__vcmpeq2(wa[i], In::kNegInf2);
      }
    }
    A += kLn2 * (acc_a.x + acc_a.y);
    if (MODE == kInterior) B += kLn2 * (acc_b.x + acc_b.y);
    viol |= v != 0;
  }

  __device__ __forceinline__ void one(int64_t, float s, float t) {
    const bool fs = s != neg_inf(), ft = t != neg_inf();
    const float lp = (s - ms) - Ls;
    const float lq = (t - mt) - Lt;
    if (MODE == kInterior) {
      float p, q, lm;
      mix_terms(lp, lq, mix, p, q, lm);
      A += ft ? q * (lq - lm) : 0.f;
      B += fs ? p * (lp - lm) : 0.f;
    } else if (MODE == kForwardKL) {  // KL(q || p)
      const float q = expd(lq);
      A += ft && fs ? q * (lq - lp) : 0.f;
      viol |= ft && !fs;
    } else {  // KL(p || q)
      const float p = expd(lp);
      A += fs && ft ? p * (lp - lq) : 0.f;
      viol |= fs && !ft;
    }
  }
  template <int N>
  __device__ __forceinline__ void vec(int64_t j, const float (&xs)[N], const float (&xt)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) one(j + i, xs[i], xt[i]);
  }
};

template <class T, int MODE>
__global__ void __maxnreg__(40) k_jsd_div(View s, View t, float beta, float* loss,
                                                      float* saved) {
  __shared__ float scratch[2 * 32];
  __shared__ int iscratch[32];
  for (int64_t r = blockIdx.x; r < s.rows; r += gridDim.x) {
    float* sv = saved + r * VPD_SAVED_PAIR;
    const RowStat st_s{sv[0], sv[1]}, st_t{sv[2], sv[3]};
    if (!stat_ok(st_s) || !stat_ok(st_t)) {
      if (threadIdx.x == 0) {
        loss[r] = qnan();
        sv[4] = qnan();
        sv[5] = qnan();
      }
      continue;
    }
    DivBody<MODE> b{st_s.m, st_s.L, st_t.m, st_t.L, {1.f - beta, beta}, 0.f, 0.f, 0};
    visit2<T>(row_ptr<T>(s, r), row_ptr<T>(t, r), s.vocab, b);
    float sums[2] = {b.A, b.B};
    block_sum<2>(sums, scratch);
    const int viol = MODE == kInterior ? 0 : block_or(b.viol, iscratch);
    if (threadIdx.x == 0) {
      if (MODE == kInterior) {
        loss[r] = beta * sums[0] + (1.f - beta) * sums[1];
        sv[4] = sums[0];
        sv[5] = sums[1];
      } else {
        const float kl = viol ? pos_inf() : sums[0];
        loss[r] = kl;
        sv[4] = MODE == kForwardKL ? kl : 0.f;
        sv[5] = MODE == kForwardKL ? 0.f : kl;
      }
    }
  }
}

// ===========================================================================
// Backward of JSD / KL: recompute p, q, ln M per element and write dS, dT.
// ===========================================================================
template <class G, int MODE>
struct BwdBody {
  float ms, Ls, mt, Lt;
  Mix mix;
  float A, B, kl;  // interior sums; endpoint KL
  float cs, ct;    // g (1 - beta), g beta (interior); g (endpoints)
  char* ds;
  char* dt;


  __device__ __forceinline__ void grads(float s, float t, float& gs, float& gt) const {
    const bool fs = s != neg_inf(), ft = t != neg_inf();
    const float lp = (s - ms) - Ls;
    const float lq = (t - mt) - Lt;
    if (MODE == kInterior) {
      float p, q, lm;
      mix_terms(lp, lq, mix, p, q, lm);
      gs = fs ? cs * p * (lp - lm - B) : 0.f;
      gt = ft ? ct * q * (lq - lm - A) : 0.f;
    } else if (MODE == kForwardKL) {  // KL(q || p): dS = g (p - q), dT = g q (lq - lp - KL)
      const float p = fs ? expd(lp) : 0.f;
      const float q = ft ? expd(lq) : 0.f;
      gs = cs * (p - q);
      gt = ft ? cs * q * (lq - lp - kl) : 0.f;
    } else {  // KL(p || q): dS = g p (lp - lq - KL), dT = g (q - p)
      const float p = fs ? expd(lp) : 0.f;
      const float q = ft ? expd(lq) : 0.f;
      gs = fs ? cs * p * (lp - lq - kl) : 0.f;
      gt = cs * (q - p);
    }
  }
  __device__ __forceinline__ void one(int64_t j, float s, float t) {
    float gs, gt;
    grads(s, t, gs, gt);
    if (ds) G::store(ds, j, gs);
    if (dt) G::store(dt, j, gt);
  }
  template <int N>
  __device__ __forceinline__ void vec(int64_t j, const float (&xs)[N], const float (&xt)[N]) {
    float gs[N], gt[N];
#pragma unroll
    for (int i = 0; i < N; ++i) grads(xs[i], xt[i], gs[i], gt[i]);
    if (ds) store_grads<G, N>(ds, j, gs, store_aligned<G::kSize, N>(ds, j));
    if (dt) store_grads<G, N>(dt, j, gt, store_aligned<G::kSize, N>(dt, j));
  }
};

template <class T, class G, int MODE>
__global__ void __launch_bounds__(kThreads) k_pair_bwd(View s, View t, float beta,
                                                       const float* grad_loss, const float* saved,
                                                       Grad ds, Grad dt) {
  for (int64_t r = blockIdx.x; r < s.rows; r += gridDim.x) {
    const float* sv = saved + r * VPD_SAVED_PAIR;
    const float A = sv[4], B = sv[5];
    const float kl = MODE == kForwardKL ? A : B;
    const bool ok = isfinite(sv[0]) && isfinite(sv[2]) &&
                    (MODE == kInterior ? (isfinite(A) && isfinite(B)) : isfinite(kl));
    char* rs = ds.data ? ds.data + r * ds.row_stride * G::kSize : nullptr;
    char* rt = dt.data ? dt.data + r * dt.row_stride * G::kSize : nullptr;
    if (!ok) {
      if (rs) zero_row<G>(rs, s.vocab);
      if (rt) zero_row<G>(rt, s.vocab);
      continue;
    }
    const float g = grad_loss ? grad_loss[r] : 1.f;
    BwdBody<G, MODE> b{sv[0], sv[1], sv[2], sv[3], {1.f - beta, beta}, A, B, kl,
                       MODE == kInterior ? g * (1.f - beta) : g, MODE == kInterior ? g * beta : g,
                       rs, rt};
    visit2<T>(row_ptr<T>(s, r), row_ptr<T>(t, r), s.vocab, b);
  }
}

// ===========================================================================
// Single-pass KL(P_a || P_b), a the target: running maxima with rescaled sums,
// W = sum_{S_a} e^{a_j - m_a} ((a_j - m_a) - (b_j - m_b)) kept relative to the
// current maxima, so KL = W / Z_a - L_a + L_b.
// ===========================================================================
struct KlAcc {
  Stat a, b;
  float w;
  int viol;
};

__device__ __forceinline__ KlAcc kl_init() { return {stat_init(), stat_init(), 0.f, 0}; }

// Re-reference a partial to the maxima (Ma, Mb); 0 if it has no a-mass.
__device__ __forceinline__ float kl_w_at(const KlAcc& x, float Ma, float Mb) {
  if (x.a.m == neg_inf() || x.b.m == neg_inf()) return 0.f;
  return exp_acc(x.a.m - Ma) * (x.w + ((Mb - x.b.m) - (Ma - x.a.m)) * x.a.z);
}

__device__ __forceinline__ KlAcc kl_merge(const KlAcc& x, const KlAcc& y) {
  KlAcc o;
  const float Ma = fmaxf(x.a.m, y.a.m), Mb = fmaxf(x.b.m, y.b.m);
  o.w = kl_w_at(x, Ma, Mb) + kl_w_at(y, Ma, Mb);
  o.a = stat_merge(x.a, y.a);
  o.b = stat_merge(x.b, y.b);
  o.viol = x.viol | y.viol;
  return o;
}

struct KlBody {
  static constexpr bool kRaw = true;
  KlAcc acc;
  // w is kept relative to both maxima (see kl_w_at); the target a weights it.
  template <class In>
  __device__ __forceinline__ void raw(int64_t, const uint4& va, const uint4& vb) {
    float2 da[4], ea[4], db[4], eb[4];
    stat_raw<In, true>(acc.b, vb, db, eb, [&](float old_m, float new_m) {
      if (old_m != neg_inf()) acc.w += (new_m - old_m) * acc.a.z;
    });
    stat_raw<In, true>(acc.a, va, da, ea, [&](float old_m, float new_m) {
      if (old_m != neg_inf()) {
        const float dd = new_m - old_m, f = exp_acc(-dd);
        acc.w = f * (acc.w - dd * acc.a.z);
      }
    });
    // sum over the pairs of e_a (d_a - d_b), in log2 units; a masked target
    // gives e_a = 0, a target with a masked other side is a support violation
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
    float2 w2 = f2(0.f);
    uint32_t viol = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w2 = fma2(ea[i], add2(da[i], neg(db[i])), w2);
      viol |= __vcmpeq2(wb[i], In::kNegInf2) & ~__vcmpeq2(wa[i], In::kNegInf2);
    }
    acc.w += kLn2 * (w2.x + w2.y);
    acc.viol |= viol != 0;
  }
  template <int N>
  __device__ __forceinline__ void vec(int64_t, const float (&xa)[N], const float (&xb)[N]) {
    float mxa = xa[0], mxb = xb[0];
#pragma unroll
    for (int i = 1; i < N; ++i) {
      mxa = fmaxf(mxa, xa[i]);
      mxb = fmaxf(mxb, xb[i]);
    }
    if (mxb > acc.b.m) {
      if (acc.b.m != neg_inf()) acc.w += (mxb - acc.b.m) * acc.a.z;
      acc.b.z *= exp_acc(acc.b.m - mxb);
      acc.b.m = mxb;
    }
    if (mxa > acc.a.m) {
      if (acc.a.m != neg_inf()) {
        const float d = mxa - acc.a.m, e = exp_acc(-d);
        acc.w = e * (acc.w - d * acc.a.z);
        acc.a.z *= e;
      }
      acc.a.m = mxa;
    }
    const float ra = stat_ref(acc.a.m), rb = stat_ref(acc.b.m);
    float za = 0.f, zb = 0.f, w = 0.f;
    int viol = 0;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float da = xa[i] - ra, db = xb[i] - rb;
      const float ea = expd(da);
      za += ea;
      zb += expd(db);
      const bool fa = xa[i] != neg_inf(), fb = xb[i] != neg_inf();
      w += fa && fb ? ea * (da - db) : 0.f;
      viol |= fa && !fb;
    }
    acc.a.z += za;
    acc.b.z += zb;
    acc.w += w;
    acc.viol |= viol;
  }
  __device__ __forceinline__ void one(int64_t j, float a, float b) {
    float xa[1] = {a}, xb[1] = {b};
    vec<1>(j, xa, xb);
  }
};

__device__ __forceinline__ KlAcc warp_kl(KlAcc x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    KlAcc y;
    y.a.m = __shfl_xor_sync(0xffffffffu, x.a.m, o);
    y.a.z = __shfl_xor_sync(0xffffffffu, x.a.z, o);
    y.b.m = __shfl_xor_sync(0xffffffffu, x.b.m, o);
    y.b.z = __shfl_xor_sync(0xffffffffu, x.b.z, o);
    y.w = __shfl_xor_sync(0xffffffffu, x.w, o);
    y.viol = __shfl_xor_sync(0xffffffffu, x.viol, o);
    x = kl_merge(x, y);
  }
  return x;
}

__device__ __forceinline__ KlAcc block_kl(KlAcc x, float* sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  x = warp_kl(x);
  __syncthreads();
  if (lane == 0) {
    sc[0 * 32 + warp] = x.a.m;
    sc[1 * 32 + warp] = x.a.z;
    sc[2 * 32 + warp] = x.b.m;
    sc[3 * 32 + warp] = x.b.z;
    sc[4 * 32 + warp] = x.w;
    sc[5 * 32 + warp] = __int_as_float(x.viol);
  }
  __syncthreads();
  KlAcc y = kl_init();
  if (lane < nw) {
    y.a = {sc[lane], sc[32 + lane]};
    y.b = {sc[64 + lane], sc[96 + lane]};
    y.w = sc[128 + lane];
    y.viol = __float_as_int(sc[160 + lane]);
  }
  y = warp_kl(y);
  __syncthreads();
  return y;
}

constexpr float kOnlineMaxLogit = 8.5070592e37f;  // 2^126

template <class T>
__global__ void __launch_bounds__(kThreads, 2) k_kl_fwd(View a, View b, Segs seg, int a_is_teacher,
                                                     float* loss, float* saved) {
  __shared__ float scratch[6 * 32];
  for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
    const char* pa = row_ptr<T>(a, r);
    const char* pb = row_ptr<T>(b, r);
    KlAcc run = kl_init();
    for (int k = 0; k < seg.count; ++k) {
      const int64_t off = seg.off[k], w = seg.off[k + 1] - off;
      KlBody body{kl_init()};
      visit2<T>(pa + off * T::kSize, pb + off * T::kSize, w, body);
      run = kl_merge(run, block_kl(body.acc, scratch));
    }
    if (threadIdx.x == 0) {
      const RowStat sa = finish_stat(run.a), sb = finish_stat(run.b);
      float kl;
      // a finite row max above 2^126 is out of contract here as on the
      // single-read kernels (the rescaling of the running sums overflows)
      if (!stat_ok(sa) || !stat_ok(sb) || sa.m > kOnlineMaxLogit || sb.m > kOnlineMaxLogit)
        kl = qnan();
      else if (run.viol)
        kl = pos_inf();
      else
        kl = run.w / run.a.z - sa.L + sb.L;
      loss[r] = kl;
      if (saved) {
        float* o = saved + r * VPD_SAVED_PAIR;
        const RowStat ss = a_is_teacher ? sb : sa, st = a_is_teacher ? sa : sb;
        o[0] = ss.m;
        o[1] = ss.L;
        o[2] = st.m;
        o[3] = st.L;
        o[4] = a_is_teacher ? kl : 0.f;
        o[5] = a_is_teacher ? 0.f : kl;
        if (isnan(kl)) o[4] = o[5] = qnan();
      }
    }
  }
}

// ===========================================================================
// Entropy: single online pass with Y = sum_S e^{x_j - m} (x_j - m) kept
// relative to the running max, H = L - Y / Z.
// ===========================================================================
struct EntAcc {
  Stat s;
  float y;
};

__device__ __forceinline__ float ent_y_at(const EntAcc& x, float M) {
  if (x.s.m == neg_inf()) return 0.f;
  return exp_acc(x.s.m - M) * (x.y - (M - x.s.m) * x.s.z);
}

__device__ __forceinline__ EntAcc ent_merge(const EntAcc& x, const EntAcc& y) {
  const float M = fmaxf(x.s.m, y.s.m);
  return {stat_merge(x.s, y.s), ent_y_at(x, M) + ent_y_at(y, M)};
}

struct EntBody {
  static constexpr bool kRaw = true;
  EntAcc acc;
  template <class In>
  __device__ __forceinline__ void raw(int64_t, const uint4& v) {
    float2 d[4], e[4];
    stat_raw<In, true>(acc.s, v, d, e, [&](float old_m, float new_m) {
      if (old_m != neg_inf()) {
        const float dd = new_m - old_m, f = exp_acc(-dd);
        acc.y = f * (acc.y - dd * acc.s.z);
      }
    });
    float2 y2 = f2(0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) y2 = fma2(e[i], d[i], y2);  // masked: e = 0, d finite
    acc.y += kLn2 * (y2.x + y2.y);
  }
  template <int N>
  __device__ __forceinline__ void vec(int64_t, const float (&x)[N]) {
    float mx = x[0];
#pragma unroll
    for (int i = 1; i < N; ++i) mx = fmaxf(mx, x[i]);
    if (mx > acc.s.m) {
      if (acc.s.m != neg_inf()) {
        const float d = mx - acc.s.m, e = exp_acc(-d);
        acc.y = e * (acc.y - d * acc.s.z);
        acc.s.z *= e;
      }
      acc.s.m = mx;
    }
    const float rf = stat_ref(acc.s.m);
    float z = 0.f, y = 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float d = x[i] - rf, e = expd(d);
      z += e;
      y += x[i] != neg_inf() ? e * d : 0.f;
    }
    acc.s.z += z;
    acc.y += y;
  }
  __device__ __forceinline__ void one(int64_t j, float v) {
    float x[1] = {v};
    vec<1>(j, x);
  }
};

__device__ __forceinline__ EntAcc block_ent(EntAcc x, float* sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    EntAcc y{{__shfl_xor_sync(0xffffffffu, x.s.m, o), __shfl_xor_sync(0xffffffffu, x.s.z, o)},
             __shfl_xor_sync(0xffffffffu, x.y, o)};
    x = ent_merge(x, y);
  }
  __syncthreads();
  if (lane == 0) {
    sc[warp] = x.s.m;
    sc[32 + warp] = x.s.z;
    sc[64 + warp] = x.y;
  }
  __syncthreads();
  EntAcc y{stat_init(), 0.f};
  if (lane < nw) y = {{sc[lane], sc[32 + lane]}, sc[64 + lane]};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    EntAcc u{{__shfl_xor_sync(0xffffffffu, y.s.m, o), __shfl_xor_sync(0xffffffffu, y.s.z, o)},
             __shfl_xor_sync(0xffffffffu, y.y, o)};
    y = ent_merge(y, u);
  }
  __syncthreads();
  return y;
}

template <class T>
__global__ void __launch_bounds__(kThreads, 3) k_entropy_fwd(View x, Segs seg, float* out, float* saved) {
  __shared__ float scratch[3 * 32];
  for (int64_t r = blockIdx.x; r < x.rows; r += gridDim.x) {
    const char* px = row_ptr<T>(x, r);
    EntAcc run{stat_init(), 0.f};
    for (int k = 0; k < seg.count; ++k) {
      const int64_t off = seg.off[k], w = seg.off[k + 1] - off;
      EntBody body{{stat_init(), 0.f}};
      visit1<T>(px + off * T::kSize, w, body);
      run = ent_merge(run, block_ent(body.acc, scratch));
    }
    if (threadIdx.x == 0) {
      const RowStat st = finish_stat(run.s);
      const float h = stat_ok(st) ? st.L - run.y / run.s.z : qnan();
      out[r] = h;
      if (saved) {
        float* o = saved + r * VPD_SAVED_ENTROPY;
        o[0] = st.m;
        o[1] = st.L;
        o[2] = h;
      }
    }
  }
}

// The same merge over the 32 lanes of a warp only (every lane gets the result).
__device__ __forceinline__ EntAcc warp_ent(EntAcc x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    EntAcc y{{__shfl_xor_sync(0xffffffffu, x.s.m, o), __shfl_xor_sync(0xffffffffu, x.s.z, o)},
             __shfl_xor_sync(0xffffffffu, x.y, o)};
    x = ent_merge(x, y);
  }
  return x;
}

// Short rows: one warp per row (each CTA of kWarpRowThreads threads holds as
// many rows as warps), so that more rows are in flight per SM than the limit of
// resident CTAs allows one CTA per row; the reductions are warp shuffles only.
template <class T>
__global__ void __maxnreg__(48) k_entropy_fwd_warp(View x, Segs seg, float* out, float* saved) {
  const int lane = threadIdx.x & 31, wpb = blockDim.x >> 5;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * wpb + (threadIdx.x >> 5); r < x.rows;
       r += static_cast<int64_t>(gridDim.x) * wpb) {
    const char* px = row_ptr<T>(x, r);
    EntAcc run{stat_init(), 0.f};
    for (int k = 0; k < seg.count; ++k) {
      const int64_t off = seg.off[k], w = seg.off[k + 1] - off;
      EntBody body{{stat_init(), 0.f}};
      visit1<T>(px + off * T::kSize, w, body, lane, 32);
      run = ent_merge(run, warp_ent(body.acc));
    }
    if (lane == 0) {
      const RowStat st = finish_stat(run.s);
      const float h = stat_ok(st) ? st.L - run.y / run.s.z : qnan();
      out[r] = h;
      if (saved) {
        float* o = saved + r * VPD_SAVED_ENTROPY;
        o[0] = st.m;
        o[1] = st.L;
        o[2] = h;
      }
    }
  }
}

template <class G>
struct EntBwdBody {
  float m, L, H, g;
  char* dx;
  __device__ __forceinline__ float grad(float x) const {
    const float lp = (x - m) - L;
    return x != neg_inf() ? -g * expd(lp) * (lp + H) : 0.f;
  }
  __device__ __forceinline__ void one(int64_t j, float x) { G::store(dx, j, grad(x)); }
  template <int N>
  __device__ __forceinline__ void vec(int64_t j, const float (&x)[N]) {
    float d[N];
#pragma unroll
    for (int i = 0; i < N; ++i) d[i] = grad(x[i]);
    store_grads<G, N>(dx, j, d, store_aligned<G::kSize, N>(dx, j));
  }
};

template <class T, class G>
__global__ void __launch_bounds__(kThreads) k_entropy_bwd(View x, const float* grad,
                                                          const float* saved, Grad dx) {
  for (int64_t r = blockIdx.x; r < x.rows; r += gridDim.x) {
    const float* sv = saved + r * VPD_SAVED_ENTROPY;
    char* rd = dx.data + r * dx.row_stride * G::kSize;
    if (!isfinite(sv[0]) || !isfinite(sv[2])) {
      zero_row<G>(rd, x.vocab);
      continue;
    }
    EntBwdBody<G> b{sv[0], sv[1], sv[2], grad ? grad[r] : 1.f, rd};
    visit1<T>(row_ptr<T>(x, r), x.vocab, b);
  }
}

// ===========================================================================
// Selected / top-k log-probabilities, and the two thin ops built on them
// ([ops page], "What"): the per-token cross-entropy at a label (-ln p_label)
// and the teacher top-k forward KL, sum_k e^{tl_k} (tl_k - ln p_{i_k}) with the
// teacher's log-probs tl at its top-k ids. An optional temperature T divides
// the logits before the softmax: the statistics are then taken of x / T (sc =
// 1 / T), in the scaled domain.
// ===========================================================================
struct StatBody {
  static constexpr bool kRaw = true;
  Stat s;
  template <class In>
  __device__ __forceinline__ void raw(int64_t, const uint4& a) {
    float2 d[4], e[4];
    stat_raw<In, false>(s, a, d, e, NoGrow{});
  }
  template <int N>
  __device__ __forceinline__ void vec(int64_t, const float (&x)[N]) {
    stat_add<N>(s, x);
  }
  __device__ __forceinline__ void one(int64_t, float x) { stat_add1(s, x); }
};

// Statistics of x / T (x * sc): (max, sum-exp) of the scaled logits.
struct ScaledStatBody {
  Stat s;
  float sc;
  template <int N>
  __device__ __forceinline__ void vec(int64_t, const float (&x)[N]) {
    float y[N];
#pragma unroll
    for (int i = 0; i < N; ++i) y[i] = x[i] * sc;
    stat_add<N>(s, y);
  }
  __device__ __forceinline__ void one(int64_t, float x) { stat_add1(s, x * sc); }
};

// What the selection computes: the log-probs themselves, the cross-entropy at
// one label per row, or the teacher top-k forward KL.
enum SelMode : int { kSelLogprobs = 0, kSelCrossEntropy = 1, kSelTopkKL = 2 };

struct Sel {
  const int64_t* index;  // [N, K]
  int K;
  int64_t ignore;
  float sc;              // 1 / T
  int mode;
  const float* tl;       // kSelTopkKL: teacher log-probs [N, K]
};

// Weight of position k of row r in the top-k KL: e^{tl}, or 0 where the id is
// ignored or the teacher has no mass.
__device__ __forceinline__ float topk_weight(const Sel& q, int64_t r, int k, int64_t i) {
  if (i == q.ignore) return 0.f;
  const float t = q.tl[r * q.K + k];
  return t == neg_inf() ? 0.f : expf(t);
}

template <class T, bool SCALED>
__global__ void __launch_bounds__(kThreads) k_select_fwd(View x, Segs seg, Sel q, float* out, float* row_out,
                                                         float* saved, int32_t* err) {
  __shared__ float scratch[64];
  for (int64_t r = blockIdx.x; r < x.rows; r += gridDim.x) {
    const char* px = row_ptr<T>(x, r);
    Stat run[1] = {stat_init()};
    for (int k = 0; k < seg.count; ++k) {
      const int64_t off = seg.off[k], w = seg.off[k + 1] - off;
      Stat part[1];
      if constexpr (SCALED) {
        ScaledStatBody body{stat_init(), q.sc};
        visit1<T>(px + off * T::kSize, w, body);
        part[0] = body.s;
      } else {
        StatBody body{stat_init()};
        visit1<T>(px + off * T::kSize, w, body);
        part[0] = body.s;
      }
      block_stat<1>(part, scratch);
      run[0] = stat_merge(run[0], part[0]);
    }
    const RowStat st = finish_stat(run[0]);  // of x * sc when SCALED
    float acc[1] = {0.f};
    for (int k = threadIdx.x; k < q.K; k += blockDim.x) {
      const int64_t i = q.index[r * q.K + k];
      float v;
      if (i == q.ignore) {
        v = 0.f;
      } else if (i < 0 || i >= x.vocab) {
        v = qnan();
        if (err) atomicExch(err, 1);
      } else if (!stat_ok(st)) {
        v = qnan();
      } else {
        const float xi = T::load(px, i);
        v = xi == neg_inf() ? neg_inf() : ((SCALED ? xi * q.sc : xi) - st.m) - st.L;
      }
      if (q.mode == kSelLogprobs) {
        out[r * q.K + k] = v;
      } else if (q.mode == kSelCrossEntropy) {
        acc[0] += -v;  // K = 1
      } else {
        const float wk = (i >= 0 && i < x.vocab) || i == q.ignore ? topk_weight(q, r, k, i) : 0.f;
        const float tk = i == q.ignore ? 0.f : q.tl[r * q.K + k];
        if (isnan(v)) acc[0] += v;
        else if (wk > 0.f) acc[0] += wk * (tk - v);  // v = -inf with teacher mass: +inf
      }
    }
    if (q.mode != kSelLogprobs) {
      block_sum<1>(acc, scratch);
      if (threadIdx.x == 0) row_out[r] = stat_ok(st) ? acc[0] : qnan();
    }
    if (saved && threadIdx.x == 0) {
      saved[r * VPD_SAVED_LOGPROBS] = st.m;
      saved[r * VPD_SAVED_LOGPROBS + 1] = st.L;
    }
  }
}

template <class G, bool SCALED>
struct LpBwdBody {
  float m, L, G_, sc;
  char* dx;
  __device__ __forceinline__ float grad(float x) const {
    if (SCALED) return x != neg_inf() ? -G_ * sc * expd((x * sc - m) - L) : 0.f;
    return x != neg_inf() ? -G_ * expd((x - m) - L) : 0.f;
  }
  __device__ __forceinline__ void one(int64_t j, float x) { G::store(dx, j, grad(x)); }
  template <int N>
  __device__ __forceinline__ void vec(int64_t j, const float (&x)[N]) {
    float d[N];
#pragma unroll
    for (int i = 0; i < N; ++i) d[i] = grad(x[i]);
    store_grads<G, N>(dx, j, d, store_aligned<G::kSize, N>(dx, j));
  }
};

template <class T, class G, bool SCALED>
__global__ void __launch_bounds__(kThreads) k_select_bwd(View x, Sel q, const float* grad, const float* saved,
                                                         Grad dx) {
  __shared__ float scratch[32];
  __shared__ int iscratch[32];
  for (int64_t r = blockIdx.x; r < x.rows; r += gridDim.x) {
    const char* px = row_ptr<T>(x, r);
    char* rd = dx.data + r * dx.row_stride * G::kSize;
    const RowStat st{saved[r * VPD_SAVED_LOGPROBS], saved[r * VPD_SAVED_LOGPROBS + 1]};
    if (!stat_ok(st)) {
      zero_row<G>(rd, x.vocab);
      continue;
    }
    // a position takes gradient when its index is valid and its log-prob finite
    auto takes = [&](int k, int64_t& i) -> bool {
      i = q.index[r * q.K + k];
      if (i == q.ignore || i < 0 || i >= x.vocab) return false;
      return T::load(px, i) != neg_inf();
    };
    // the upstream gradient of position k
    auto up = [&](int k, int64_t i) -> float {
      if (q.mode == kSelLogprobs) return grad ? grad[r * q.K + k] : 1.f;
      const float g = grad ? grad[r] : 1.f;
      if (q.mode == kSelCrossEntropy) return -g;
      return -g * topk_weight(q, r, k, i);
    };
    if (q.mode == kSelTopkKL) {
      // +inf KL (an id the teacher gives mass that the student masks): no gradient
      int inf_row = 0;
      for (int k = threadIdx.x; k < q.K; k += blockDim.x) {
        const int64_t i = q.index[r * q.K + k];
        if (i != q.ignore && i >= 0 && i < x.vocab && topk_weight(q, r, k, i) > 0.f && T::load(px, i) == neg_inf())
          inf_row = 1;
      }
      if (block_or(inf_row, iscratch)) {
        zero_row<G>(rd, x.vocab);
        continue;
      }
    }
    float gsum[1] = {0.f};
    for (int k = threadIdx.x; k < q.K; k += blockDim.x) {
      int64_t i;
      if (takes(k, i)) gsum[0] += up(k, i);
    }
    block_sum<1>(gsum, scratch);
    LpBwdBody<G, SCALED> b{st.m, st.L, gsum[0], q.sc, rd};
    visit1<T>(px, x.vocab, b);
    __syncthreads();
    // the selected tokens: the sum of their upstream gradients minus p_j G (times sc)
    for (int k = threadIdx.x; k < q.K; k += blockDim.x) {
      int64_t i;
      if (!takes(k, i)) continue;
      bool first = true;
      float gi = 0.f;
      for (int k2 = 0; k2 < q.K; ++k2) {
        int64_t i2;
        if (!takes(k2, i2) || i2 != i) continue;
        if (k2 < k) {
          first = false;
          break;
        }
        gi += up(k2, i2);
      }
      if (first) G::store(rd, i, (SCALED ? q.sc : 1.f) * gi + b.grad(T::load(px, i)));
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Launch helpers.
// ---------------------------------------------------------------------------
// Threads per CTA for rows of `vocab` elements of `esize` bytes. Kernels that
// write a gradient row: about 16 16-byte vectors per thread, a multiple of 64
// from 64 to kThreads. Kernels that only reduce a row (statistics,
// divergence, KL and entropy forwards, selections): about 256 vectors per
// thread, a multiple of 32 from 32 to kThreads, so that many rows are in
// flight on each SM and each row's latency overlaps the others' (measured at
// V = 151936: entropy forward 0.533 -> 0.400 ms, online KL forward 1.353 ->
// 1.200 ms, two-pass JSD forward 1.805 -> 1.579 ms; at V = 16032 entropy
// forward 0.084 -> 0.062 ms; the backward kernels are slower with fewer
// threads per row).
int threads_for(int64_t vocab, int esize, bool reduce_only = false) {
  const int64_t nv = vocab * esize / 16;
  if (reduce_only) {
    const int64_t t = (nv / 256 + 31) / 32 * 32;
    return t < 32 ? 32 : (t > kThreads ? kThreads : static_cast<int>(t));
  }
  const int64_t t = (nv / 16 + 63) / 64 * 64;
  return t < 64 ? 64 : (t > kThreads ? kThreads : static_cast<int>(t));
}

// SMs a launch may fill on this thread, when set (0: all of them): the rows a
// fused launch hands to the SMs its clusters leave idle run on as many CTAs as
// fit that many SMs.
thread_local int g_grid_cap = 0;

template <class Kern>
int grid_for(Kern kernel, int64_t rows, int threads) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int sms = g_grid_cap > 0 && g_grid_cap < sm_count() ? g_grid_cap : sm_count();
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  return static_cast<int>(rows < cap ? rows : cap);
}

// One CTA per row at a time (grid-stride over rows), `threads` per CTA.
template <class Kern, class... Args>
cudaError_t launch_rows(Kern kernel, int64_t rows, int threads, cudaStream_t stream, Args... args) {
  if (rows <= 0) return cudaSuccess;
  kernel<<<grid_for(kernel, rows, threads), threads, 0, stream>>>(args...);
  note_launch();
  return cudaGetLastError();
}

// One warp per row at a time (grid-stride over groups of rows), CTAs of
// kWarpRowThreads threads.
constexpr int kWarpRowThreads = 128;
template <class Kern, class... Args>
cudaError_t launch_warp_rows(Kern kernel, int64_t rows, cudaStream_t stream, Args... args) {
  if (rows <= 0) return cudaSuccess;
  constexpr int wpb = kWarpRowThreads / 32;
  kernel<<<grid_for(kernel, (rows + wpb - 1) / wpb, kWarpRowThreads), kWarpRowThreads, 0, stream>>>(args...);
  note_launch();
  return cudaGetLastError();
}

template <template <class> class F, class... Args>
cudaError_t by_input(int dtype, Args&&... args) {
  switch (dtype) {
    case kF32: return F<F32>::run(args...);
    case kBF16: return F<BF16>::run(args...);
    case kF16: return F<F16>::run(args...);
  }
  return cudaErrorInvalidValue;
}

template <class T, template <class, class> class F, class... Args>
cudaError_t by_grad(int gdtype, Args&&... args) {
  switch (gdtype) {
    case kF32: return F<T, GF32>::run(args...);
    case kBF16: return F<T, GBF16>::run(args...);
    case kF16: return F<T, GF16>::run(args...);
  }
  return cudaErrorInvalidValue;
}

template <class T>
struct PairStatsL {
  static cudaError_t run(const View& s, const View& t, const Segs& seg, float* saved, cudaStream_t st) {
    return launch_rows(k_pair_stats<T>, s.rows, threads_for(s.vocab, T::kSize, true), st, s, t, seg, saved);
  }
};

template <class T>
struct DivL {
  static cudaError_t run(const View& s, const View& t, double beta, float* loss, float* saved,
                         cudaStream_t st) {
    const float b = static_cast<float>(beta);
    if (beta == 0.0) return launch_rows(k_jsd_div<T, kForwardKL>, s.rows, threads_for(s.vocab, T::kSize, true), st, s, t, b, loss, saved);
    if (beta == 1.0) return launch_rows(k_jsd_div<T, kReverseKL>, s.rows, threads_for(s.vocab, T::kSize, true), st, s, t, b, loss, saved);
    return launch_rows(k_jsd_div<T, kInterior>, s.rows, threads_for(s.vocab, T::kSize, true), st, s, t, b, loss, saved);
  }
};

template <class T, class G>
struct BwdL {
  static cudaError_t run(const View& s, const View& t, double beta, const float* g,
                         const float* saved, const Grad& ds, const Grad& dt, cudaStream_t st) {
    const float b = static_cast<float>(beta);
    if (beta == 0.0)
      return launch_rows(k_pair_bwd<T, G, kForwardKL>, s.rows, threads_for(s.vocab, T::kSize), st, s, t, b, g, saved, ds, dt);
    if (beta == 1.0)
      return launch_rows(k_pair_bwd<T, G, kReverseKL>, s.rows, threads_for(s.vocab, T::kSize), st, s, t, b, g, saved, ds, dt);
    return launch_rows(k_pair_bwd<T, G, kInterior>, s.rows, threads_for(s.vocab, T::kSize), st, s, t, b, g, saved, ds, dt);
  }
};

template <class T>
struct BwdByGrad {
  static cudaError_t run(const View& s, const View& t, double beta, const float* g,
                         const float* saved, const Grad& ds, const Grad& dt, cudaStream_t st) {
    const int gd = ds.data ? ds.dtype : dt.dtype;
    return by_grad<T, BwdL>(gd, s, t, beta, g, saved, ds, dt, st);
  }
};

template <class T>
struct KlL {
  static cudaError_t run(const View& a, const View& b, const Segs& seg, int a_is_teacher, float* loss,
                         float* saved, cudaStream_t st) {
    return launch_rows(k_kl_fwd<T>, a.rows, threads_for(a.vocab, T::kSize, true), st, a, b, seg, a_is_teacher, loss, saved);
  }
};

template <class T>
struct EntL {
  static cudaError_t run(const View& x, const Segs& seg, float* out, float* saved, cudaStream_t st) {
    const int threads = threads_for(x.vocab, T::kSize, true);
    if (threads == 32)  // short rows: one warp per row
      return launch_warp_rows(k_entropy_fwd_warp<T>, x.rows, st, x, seg, out, saved);
    return launch_rows(k_entropy_fwd<T>, x.rows, threads, st, x, seg, out, saved);
  }
};

template <class T, class G>
struct EntBwdL {
  static cudaError_t run(const View& x, const float* g, const float* saved, const Grad& dx,
                         cudaStream_t st) {
    return launch_rows(k_entropy_bwd<T, G>, x.rows, threads_for(x.vocab, T::kSize), st, x, g, saved, dx);
  }
};

template <class T>
struct EntBwdByGrad {
  static cudaError_t run(const View& x, const float* g, const float* saved, const Grad& dx,
                         cudaStream_t st) {
    return by_grad<T, EntBwdL>(dx.dtype, x, g, saved, dx, st);
  }
};

template <class T>
struct SelL {
  static cudaError_t run(const View& x, const Segs& seg, const Sel& q, float* out, float* row_out, float* saved,
                         int32_t* err, cudaStream_t st) {
    if (q.sc != 1.f)
      return launch_rows(k_select_fwd<T, true>, x.rows, threads_for(x.vocab, T::kSize, true), st, x, seg, q, out, row_out,
                         saved, err);
    return launch_rows(k_select_fwd<T, false>, x.rows, threads_for(x.vocab, T::kSize, true), st, x, seg, q, out, row_out,
                       saved, err);
  }
};

template <class T, class G>
struct SelBwdL {
  static cudaError_t run(const View& x, const Sel& q, const float* g, const float* saved, const Grad& dx,
                         cudaStream_t st) {
    if (q.sc != 1.f)
      return launch_rows(k_select_bwd<T, G, true>, x.rows, threads_for(x.vocab, T::kSize), st, x, q, g, saved, dx);
    return launch_rows(k_select_bwd<T, G, false>, x.rows, threads_for(x.vocab, T::kSize), st, x, q, g, saved, dx);
  }
};

template <class T>
struct SelBwdByGrad {
  static cudaError_t run(const View& x, const Sel& q, const float* g, const float* saved, const Grad& dx,
                         cudaStream_t st) {
    return by_grad<T, SelBwdL>(dx.dtype, x, q, g, saved, dx, st);
  }
};

std::atomic<uint64_t> g_launches{0};

}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

GridCap::GridCap(int ctas) : prev_(g_grid_cap) { g_grid_cap = ctas; }
GridCap::~GridCap() { g_grid_cap = prev_; }
uint64_t launch_count() { return g_launches.load(std::memory_order_relaxed); }

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 1;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n < 1) n = 1;
  if (dev < 64) cache[dev] = n;
  return n;
}

cudaError_t launch_pair_stats(const View& s, const View& t, const Segs& seg, float* saved,
                              cudaStream_t stream) {
  return by_input<PairStatsL>(s.dtype, s, t, seg, saved, stream);
}

cudaError_t launch_jsd_div(const View& s, const View& t, double beta, float* loss, float* saved,
                           cudaStream_t stream) {
  return by_input<DivL>(s.dtype, s, t, beta, loss, saved, stream);
}

cudaError_t launch_pair_bwd(const View& s, const View& t, double beta, const float* grad_loss,
                            const float* saved, const Grad& ds, const Grad& dt, cudaStream_t stream) {
  if (!ds.data && !dt.data) return cudaSuccess;
  return by_input<BwdByGrad>(s.dtype, s, t, beta, grad_loss, saved, ds, dt, stream);
}

cudaError_t launch_kl_fwd(const View& s, const View& t, int reverse, const Segs& seg, float* loss,
                          float* saved, cudaStream_t stream) {
  // reverse = 0: KL(P_t || P_s), the teacher is the target
  if (reverse) return by_input<KlL>(s.dtype, s, t, seg, 0, loss, saved, stream);
  return by_input<KlL>(s.dtype, t, s, seg, 1, loss, saved, stream);
}

cudaError_t launch_entropy_fwd(const View& x, const Segs& seg, float* out, float* saved,
                               cudaStream_t stream) {
  return by_input<EntL>(x.dtype, x, seg, out, saved, stream);
}

cudaError_t launch_entropy_bwd(const View& x, const float* grad, const float* saved, const Grad& dx,
                               cudaStream_t stream) {
  return by_input<EntBwdByGrad>(x.dtype, x, grad, saved, dx, stream);
}

cudaError_t launch_select_fwd(const View& x, const Segs& seg, const int64_t* index, int k, int64_t ignore_index,
                              float inv_temperature, int mode, const float* teacher_logp, float* out,
                              float* row_out, float* saved, int32_t* err_flag, cudaStream_t stream) {
  const Sel q{index, k, ignore_index, inv_temperature, mode, teacher_logp};
  return by_input<SelL>(x.dtype, x, seg, q, out, row_out, saved, err_flag, stream);
}

cudaError_t launch_select_bwd(const View& x, const int64_t* index, int k, int64_t ignore_index,
                              float inv_temperature, int mode, const float* teacher_logp, const float* grad,
                              const float* saved, const Grad& dx, cudaStream_t stream) {
  const Sel q{index, k, ignore_index, inv_temperature, mode, teacher_logp};
  return by_input<SelBwdByGrad>(x.dtype, x, q, grad, saved, dx, stream);
}

}  // namespace vpd
