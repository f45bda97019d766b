// common.cuh -- device helpers shared by the attention kernels (sm_103a).
//
// Inline-PTX wrappers for mbarriers, TMA tiled loads, tcgen05 (MMA, TMEM
// alloc / ld / st, commit, fences) and mma.sync, the bounded waits every
// kernel uses, element conversions, and the visibility predicate.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// ----------------------------------------------------------------- params
// Everything a kernel needs to know about one attention call.  Pointers are
// device pointers; layouts follow include/attn.h.
struct Params {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    const void* o_in;    // backward: forward output
    const void* dout;    // backward: dO
    const float* lse_in; // backward: saved LSE
    void* dq;
    void* dk;
    void* dv;
    float* ndelta;       // backward: -D = -rowsum(dO*O)     [B*H][tq_pad]
    float* nlse2;        // backward: -LSE*log2(e), -inf where LSE = -inf  [B*H][tq_pad]
    int tq_pad;          // backward: Tq rounded up to 64 (row stride of ndelta / nlse2)
    int kv_chunk;        // backward dK/dV: (batch, KV head) pairs whose key blocks are numbered together (0: all)
    float* ws;           // decode: split partials
    const float* key_mask;
    long long mask_bstride;
    int B, Tq, Tk, H, Hkv, hd, G;
    float scale;         // softmax scale (natural units)
    float scale_log2;    // scale * log2(e)
    int wl, wr;          // visible keys [p - wl, p + wr] for the query at position p; -1: unbounded side
    // additive score bias, bias[b*bias_sb + h*bias_sh + i*bias_sq + j*bias_sk], or NULL
    const float* bias;
    long long bias_sb, bias_sh, bias_sq, bias_sk;
    float softcap;       // 0 = off
    int q_offset;
    int splits, chunk;   // decode
    const int* lengths;  // decode: per-batch valid cache length on the device, or NULL (Tk for all)
    // Packed variable-length batches: sequence b owns query rows [cu_q[b], cu_q[b+1])
    // and key rows [cu_k[b], cu_k[b+1]) of one packed tensor (device int32 prefix
    // sums, B+1 each); Tq and Tk then bound the sequence lengths.  NULL: dense [B][T].
    const int* cu_q;
    const int* cu_k;
    int total_q, total_k;  // packed: rows of q/o and of k/v (no access goes past them)
    // rotary embedding of the query tiles inside the forward (or NULL): cosine and
    // sine of rotary position s (query row i sits at s = q_offset + i) and pair
    // index c at rope_tab[2 * (c * rope_npos + s)], [+1]; rope_npos positions
    const float* rope_tab;
    int rope_npos;
    // Packed fused-QKV rows (one batch, Tq = Tk, q_offset 0), or NULL: row r sees only
    // keys j in [row_bounds[r].x, row_bounds[r].y), its own sequence (a range holding r;
    // the sequences lie back to back, so the bounds never decrease down the rows).  The
    // window then applies inside the sequence.
    const int2* row_bounds;
    // With row_bounds, the order in which the work items' row blocks run (heaviest
    // first: a permutation of the blocks of 256 rows in the forward, of 128 rows in the
    // backward), or NULL for the plain order.  It decides only which CTA takes which
    // block when; every block is computed the same way.
    const int* item_order;
    unsigned int* status;
};

// Status word bits (which wait ran out).
enum : unsigned int {
    ST_FWD_PRODUCER = 1u << 0,
    ST_FWD_MMA = 1u << 1,
    ST_FWD_SOFTMAX = 1u << 2,
    ST_BWD_PRODUCER = 1u << 3,
    ST_BWD_MMA = 1u << 4,
    ST_BWD_COMPUTE = 1u << 5,
    ST_DEC_WAIT = 1u << 6,
    ST_SELFTEST = 1u << 7,
    ST_TEARDOWN = 1u << 8,
    ST_VARLEN_BOUNDS = 1u << 9,  // a packed sequence longer than the bound, or cu_seqlens decreasing
};

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s: no wait is ever that long

// ------------------------------------------------------------- conversions
template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float to_f(float x) { return x; }
    static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct Elem<__half> {
    static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
    static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// pack two floats into one 32-bit word of two 16-bit values (lo = first)
template <bool BF16> __device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<true>(float lo, float hi) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
}
template <> __device__ __forceinline__ uint32_t pack2<false>(float lo, float hi) {
    __half2 t = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
}
// dot product of two words of two 16-bit values each, in fp32
template <bool BF16> __device__ __forceinline__ float dot2(uint32_t a, uint32_t b);
template <> __device__ __forceinline__ float dot2<true>(uint32_t a, uint32_t b) {
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a));
    const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b));
    return fmaf(x.x, y.x, x.y * y.y);
}
template <> __device__ __forceinline__ float dot2<false>(uint32_t a, uint32_t b) {
    const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&a));
    const float2 y = __half22float2(*reinterpret_cast<const __half2*>(&b));
    return fmaf(x.x, y.x, x.y * y.y);
}

// --------------------------------------------------------------- sequences
// Where sequence b's rows live.  Dense: batch b of [B][T] tensors.  Packed:
// rows q0 .. q0+tq-1 (queries) and k0 .. k0+tk-1 (keys) of the single packed
// batch.  zb is the batch coordinate of the 3-D tensor maps; the linear row of
// query i is zb*Tq + q0 + i (keys: zb*Tk + k0 + j).  A packed sequence longer
// than the launch bound or running past the tensor's rows (or a decreasing or
// negative prefix sum) is cut to what fits (or to nothing) and flags
// ST_VARLEN_BOUNDS, so that no access leaves the caller's buffers.
struct Seq {
    int q0, tq, k0, tk, zb;
};
template <bool kPacked>
__device__ __forceinline__ Seq seq_of(const Params& P, int b) {
    Seq s;
    if constexpr (kPacked) {
        const int a0 = __ldg(P.cu_q + b), a1 = __ldg(P.cu_q + b + 1);
        const int c0 = __ldg(P.cu_k + b), c1 = __ldg(P.cu_k + b + 1);
        const bool start_ok = a0 >= 0 && c0 >= 0 && a0 <= P.total_q && c0 <= P.total_k;
        s.q0 = start_ok ? a0 : 0;
        s.k0 = start_ok ? c0 : 0;
        s.tq = start_ok ? min(min(max(a1 - a0, 0), P.Tq), P.total_q - a0) : 0;
        s.tk = start_ok ? min(min(max(c1 - c0, 0), P.Tk), P.total_k - c0) : 0;
        s.zb = 0;
        if ((a1 - a0 != s.tq || c1 - c0 != s.tk) && P.status) atomicOr(P.status, ST_VARLEN_BOUNDS);
    } else {
        s.q0 = 0;
        s.k0 = 0;
        s.tq = P.Tq;
        s.tk = P.Tk;
        s.zb = b;
    }
    return s;
}
// the same, choosing the layout at run time (the CUDA-core kernels)
__device__ __forceinline__ Seq seq_any(const Params& P, int b) {
    return P.cu_q ? seq_of<true>(P, b) : seq_of<false>(P, b);
}

// ------------------------------------------------------------ rotary turn
// Rotate-half RoPE turn of the pair (a, b) = (x[i], x[i + hd/2]) by the angle whose
// cosine and sine are c and s (the inverse turn passes -s).  Written out with fmaf
// so that every kernel that rotates (the standalone pass, the forward's Q tiles)
// rounds alike.
__device__ __forceinline__ void rope_turn(float a, float b, float c, float s, float& lo, float& hi) {
    lo = fmaf(a, c, -(b * s));
    hi = fmaf(b, c, a * s);
}

// ------------------------------------------------------------ visibility
// Keys [x, y) that packed fused-QKV row r may see by its sequence bounds, clamped to
// [0, n) so that no access leaves the rows.
__device__ __forceinline__ int2 row_keys(const Params& P, int r, int n) {
    const int2 rb = __ldg(P.row_bounds + r);
    return make_int2(max(rb.x, 0), min(rb.y, n));
}

// Key j (of tk) visible to the query at absolute position p (see include/attn.h).
__device__ __forceinline__ bool visible(const Params& P, int b, int p, int j, int tk) {
    if (j < 0 || j >= tk) return false;
    if (P.row_bounds) {  // packed fused-QKV rows: position p is row p of the one batch
        const int2 rk = row_keys(P, p, tk);
        if (j < rk.x || j >= rk.y) return false;
    }
    if (P.wr >= 0 && j > p + P.wr) return false;
    if (P.wl >= 0 && j < p - P.wl) return false;
    if (P.key_mask && !(P.key_mask[(long long)b * P.mask_bstride + j] > 0.5f)) return false;
    return true;
}

// Keys of batch b that a key mask can keep: [lo, hi) covers every key j < tk with
// mask > 0.5 (lo = hi when there is none).  Called by a whole warp: lane l scans its
// own stretch of ceil(tk/32) keys, and the stretches holding a kept key bound the
// span, so the result may include masked keys at its ends but never leaves a kept
// key out.  Kernels use it to skip key tiles a prefix (or suffix) mask removes.
__device__ __forceinline__ int2 mask_span(const Params& P, int b, int tk) {
    const int lane = threadIdx.x & 31;
    const int seg = (tk + 127) / 128 * 4;  // a multiple of 4 keys per lane
    const float* row = P.key_mask + (long long)b * P.mask_bstride;
    bool any = false;
    const int j0 = lane * seg, j1 = min(tk, j0 + seg);
    // independent loads (no early exit), four keys at a time when the row allows
    if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0 && j1 - j0 == seg) {
        const float4* r4 = reinterpret_cast<const float4*>(row + j0);
        for (int e = 0; e < seg / 4; ++e) {
            const float4 m = __ldg(r4 + e);
            any = any || (m.x > 0.5f) || (m.y > 0.5f) || (m.z > 0.5f) || (m.w > 0.5f);
        }
    } else {
        for (int j = j0; j < j1; ++j) any = any || (__ldg(row + j) > 0.5f);
    }
    const unsigned bal = __ballot_sync(0xffffffffu, any);
    if (bal == 0u) return make_int2(0, 0);
    const int first = __ffs(bal) - 1, last = 31 - __clz(bal);
    return make_int2(first * seg, min(tk, (last + 1) * seg));
}
constexpr int kMaskSpanMax = 64;  // batches whose spans a kernel keeps in shared memory
// packed batches of at most this many sequences get compact item numberings (one lane
// per sequence)
constexpr int kVlCompact = 32;

// Range of keys [lo, hi) that any query with position in [p0, p1] can see,
// before the key mask: the window [p - wl, p + wr] (-1 = unbounded side).
__host__ __device__ __forceinline__ void key_range(int wl, int wr, int Tk, int p0, int p1, int* lo, int* hi) {
    long long l = 0, h = Tk;
    if (wr >= 0 && (long long)p1 + wr + 1 < h) h = (long long)p1 + wr + 1;
    if (wl >= 0 && (long long)p0 - wl > l) l = (long long)p0 - wl;
    if (h < l) h = l;
    *lo = (int)l;
    *hi = (int)h;
}

// True when every query in [p0, p1] sees every key in [j0, j1) (ignoring the key mask).
__host__ __device__ __forceinline__ bool tile_full(int wl, int wr, int Tk, int p0, int p1, int j0, int j1) {
    if (j1 > Tk) return false;
    if (wr >= 0 && (long long)j1 - 1 > (long long)p0 + wr) return false;  // newest key ahead of the oldest query
    if (wl >= 0 && (long long)j0 < (long long)p1 - wl) return false;      // oldest key behind the newest query
    return true;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fast_rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// tanh(x) = 1 - 2/(exp(2x)+1), with exp(2x) = 2^(2x*log2 e).  Absolute error
// a few ulp of 1, which is what softcap * tanh needs (the product's error is
// softcap * 1e-7).  Saturates correctly for large |x|.
__device__ __forceinline__ float tanh_accurate(float x) {
    float e = fast_exp2(x * 2.8853900817779268f);  // 2*log2(e)
    return 1.0f - 2.0f * fast_rcp(e + 1.0f);
}

// softcap * tanh(y) for small |y| without the two MUFU operations of
// tanh_accurate: tanh(y) = y * (1 + t * R(t)), t = y^2, R a cubic fitted to
// (tanh(y)/y - 1)/t on |y| <= kTanhPolyY (weighted least squares on Chebyshev
// nodes, weights chosen for the relative error of tanh; that error stays below
// 2e-8 there, under fp32 rounding).  Callers check the range and fall back to
// tanh_accurate for larger |y|.  The leading coefficient is positive, so a
// score of -inf still maps to -inf through every form built on it below.
constexpr float kTanhPolyY = 0.5f;
constexpr float kTanhR0 = -0.3333313623f, kTanhR1 = 0.1332571191f, kTanhR2 = -0.0530346934f,
                kTanhR3 = 0.0172199592f;

// ------------------------------------------------- packed fp32 pairs (f32x2)
// The sm_100 family issues add/mul/fma on two fp32 values held in one 64-bit
// register as one instruction.
__device__ __forceinline__ uint64_t f2_make(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t a, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Per-launch constants of the softcapped score for a raw score r = q.k, with
// c = scale/softcap: tanh(c*r) = c*g, g = r + r*u*S(u), u = r^2 and
// S(u) = c^2*R(c^2*u).  The capped score in log2 units is then sl2*g
// (sl2 = scale*log2 e) and the softcap derivative 1 - c^2*g^2.
struct CapPoly {
    uint64_t s0, s1, s2, s3;  // S's coefficients, both halves equal
    uint64_t nc2;             // -c^2, both halves
    float u_max, r_max;       // the polynomial serves u <= u_max, i.e. |r| <= r_max
    bool inf_ok;              // S(+inf) = +inf, so a -inf score stays -inf through g
};
__device__ __forceinline__ CapPoly cap_poly(float scale, float softcap) {
    const float c = scale / fmaxf(softcap, 1e-30f), c2 = c * c;
    const float k0 = c2 * kTanhR0, k1 = c2 * c2 * kTanhR1, k2 = c2 * c2 * c2 * kTanhR2,
                k3 = c2 * c2 * c2 * c2 * kTanhR3;
    CapPoly cp;
    cp.s0 = f2_make(k0, k0);
    cp.s1 = f2_make(k1, k1);
    cp.s2 = f2_make(k2, k2);
    cp.s3 = f2_make(k3, k3);
    cp.nc2 = f2_make(-c2, -c2);
    cp.r_max = fminf(kTanhPolyY / c, 1e18f);
    cp.u_max = cp.r_max * cp.r_max;
    cp.inf_ok = k3 > 0.f;
    return cp;
}
// g of a pair of raw scores (see CapPoly)
__device__ __forceinline__ uint64_t cap_g(const CapPoly& cp, uint64_t r, uint64_t& u) {
    u = f2_mul(r, r);
    uint64_t sp = f2_fma(u, cp.s3, cp.s2);
    sp = f2_fma(u, sp, cp.s1);
    sp = f2_fma(u, sp, cp.s0);
    return f2_fma(r, f2_mul(u, sp), r);
}

// A shorter softcap polynomial for tiles whose scores all lie well inside the
// fitted polynomial's range: tanh(y) = y * (1 + t * (kTanhS0 + kTanhS1 * t)),
// t = y^2, for |y| <= kTanhShortY (weighted least squares on Chebyshev nodes for
// the relative error of tanh, below 1e-8 there in exact arithmetic).  Two
// fewer packed operations per pair of scores than the cubic R.  The leading
// coefficient is positive, so a score of -inf still maps to -inf.
constexpr float kTanhShortY = 0.125f;
constexpr float kTanhS0 = -0.3333277106f, kTanhS1 = 0.1321673691f;
struct CapShort {
    uint64_t s0, s1;  // S(u) = c^2*kTanhS0 + c^4*kTanhS1*u, both halves equal (c = scale/softcap)
    float r_max;      // the polynomial serves raw scores |r| <= r_max
    bool inf_ok;      // -inf maps to -inf (c^4*kTanhS1 did not underflow)
};
__device__ __forceinline__ CapShort cap_short(float scale, float softcap) {
    const float c = scale / fmaxf(softcap, 1e-30f), c2 = c * c;
    const float k0 = c2 * kTanhS0, k1 = c2 * c2 * kTanhS1;
    CapShort cs;
    cs.s0 = f2_make(k0, k0);
    cs.s1 = f2_make(k1, k1);
    cs.r_max = fminf(kTanhShortY / c, 1e18f);
    cs.inf_ok = k1 > 0.f;
    return cs;
}
// g = r + r*u*S(u), u = r^2, of a pair of raw scores: tanh(c*r) = c*g
__device__ __forceinline__ uint64_t cap_g_short(const CapShort& cs, uint64_t r) {
    const uint64_t u = f2_mul(r, r);
    return f2_fma(r, f2_mul(u, f2_fma(u, cs.s1, cs.s0)), r);
}

// --------------------------------------------------------------- timing
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Non-blocking probe of a phase (no suspend): the cheap path when it already completed.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: true when the phase of the given parity completed, false
// (and the status bit set) after the time limit or when *abort is raised.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int* status,
                                          unsigned int code, volatile int* abort_flag) {
    if (mbar_test_wait(bar, parity)) return true;
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
#pragma unroll 1
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag && *abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(status, code);
            if (abort_flag) *abort_flag = 1;
            return false;
        }
    }
}

// The k-th work item of this CTA in a persistent kernel: rounds of gridDim.x
// items taken alternately in CTA order and reversed, so that with items numbered
// longest first each CTA pairs heavier items with lighter ones.
__device__ __forceinline__ int snake_item(int k) {
    const int g = (int)gridDim.x, c = (int)blockIdx.x;
    return k * g + ((k & 1) ? g - 1 - c : c);
}

// Bounded wait until a shared counter reaches target (an execution order only:
// no data is published through it).  Sleeps briefly between polls so that the
// waiting warps leave issue slots to the warps they wait for.
__device__ __forceinline__ bool count_wait(const int* counter, int target, unsigned int* status, unsigned int code,
                                           volatile int* abort_flag) {
    const volatile int* cc = counter;
    if (*cc >= target) return true;
    const unsigned long long t0 = globaltimer();
#pragma unroll 1
    while (true) {
        __nanosleep(20);
        if (*cc >= target) return true;
        if (abort_flag && *abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(status, code);
            if (abort_flag) *abort_flag = 1;
            return false;
        }
    }
}

// Bounded wait by a whole warp; true only when every lane saw the phase.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, unsigned int* status, unsigned int code,
                                          volatile int* abort_flag) {
    const bool r = mbar_wait(bar, parity, status, code, abort_flag);
    return __all_sync(0xffffffffu, r);
}

// True in exactly one lane of the (converged, full) warp, the same lane every
// time.  Issuing tcgen05.mma / tcgen05.commit / TMA this way from a warp that
// runs the issue loop together keeps the operand arithmetic warp-uniform; the
// issue then costs about a third of the same loop run by a single lane.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int c0, int c1, int c2, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}
// Tiled store shared -> global through a tensor map (coordinates as for the load;
// rows outside the map are not written).  Completion is tracked by bulk groups of
// the issuing thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
// 4-D forms, for maps over [batches][rows][heads][hd] (padded head sizes: the
// box's 64 columns reach past hd, those columns load as zeros and are not stored)
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}
// Activation tiles: box bx (64 columns) of head h, rows from `row`, batch zb.  With
// kPad the map is 4-D ([zb][row][h][col], hd < the kernel's padded head size), else
// 3-D ([zb][row][h*HD + col]).
template <bool kPad, int HD>
__device__ __forceinline__ void tile_load(uint32_t dst, const CUtensorMap* map, uint32_t bar, int h, int bx, int row,
                                          int zb) {
    if constexpr (kPad) tma_load_4d(dst, map, bar, bx * 64, h, row, zb);
    else tma_load_3d(dst, map, bar, h * HD + bx * 64, row, zb);
}
template <bool kPad, int HD>
__device__ __forceinline__ void tile_store(const CUtensorMap* map, uint32_t src, int h, int col, int row, int zb) {
    if constexpr (kPad) tma_store_4d(map, src, col, h, row, zb);
    else tma_store_3d(map, src, h * HD + col, row, zb);
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's bulk stores are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
// generic-proxy writes to shared memory become visible to the async (TMA) proxy
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tcgen05
// Instruction descriptor for kind::f16 with fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int M, int N, bool a_mn_major,
                                                 bool b_mn_major) {
    return (1u << 4)                                  // D format: f32
           | ((bf16 ? 1u : 0u) << 7)                  // A format: bf16 / f16
           | ((bf16 ? 1u : 0u) << 10)                 // B format
           | ((a_mn_major ? 1u : 0u) << 15)           // A major (0 = K-major)
           | ((b_mn_major ? 1u : 0u) << 16)           // B major
           | ((uint32_t)(N >> 3) << 17)               // N / 8
           | ((uint32_t)(M >> 4) << 24);              // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle, atoms 1024-byte aligned.
//   K-major  : rows of 128 B (64 x 16-bit), SBO = stride of 8-row groups.
//   MN-major : LBO = stride between 64-element MN chunks, SBO = 8-row K groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;  // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on an mbarrier when every tcgen05 op this thread issued so far completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// The same three issued by one lane of a converged warp, chosen by elect.sync: the
// elect predicate guards the single-thread instruction itself, so the warp takes no
// branch (and needs no reconvergence) around each issue.  Call from the whole warp.
__device__ __forceinline__ void mma_ss_e(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts_e(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit_e(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// 32 lanes x 32 columns of 32-bit TMEM -> 32 registers per thread (its lane).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// Wait for outstanding tcgen05.ld, then pin the registers after the wait so
// no use of them is scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31]));
}
__device__ __forceinline__ void tmem_ld_wait_only() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_pin(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31]));
}
// 32 registers per thread -> 32 lanes x 32 columns of TMEM.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
// 16 registers per thread -> 32 lanes x 16 columns of TMEM.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Warpgroup register reallocation (all 128 threads of the warpgroup execute it).
template <int N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Named barrier among `nthreads` threads (multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- mma.sync
// m16n8k16, 16-bit inputs, fp32 accumulate (used by the decode kernel).
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    if constexpr (BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Offset of 16-byte chunk `c` (0..7) of row `r` inside a 128-byte-swizzled
// tile whose rows are 128 bytes (the layout TMA writes with SWIZZLE_128B).
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c) {
    return r * 128u + ((c ^ (r & 7u)) << 4);
}

}  // namespace attn

namespace attn {
// Queries [lo, hi) (row indices) that can see at least one key of [j0, j1),
// before the key mask: position p = i + q_offset with j0 - wr <= p <= j1 - 1 + wl.
__host__ __device__ __forceinline__ void query_range(int wl, int wr, int Tq, int q_offset, int j0, int j1, int* lo,
                                                     int* hi) {
    long long l = 0, h = Tq;
    if (wr >= 0 && (long long)j0 - wr - q_offset > l) l = (long long)j0 - wr - q_offset;
    if (wl >= 0 && (long long)j1 - 1 + wl - q_offset + 1 < h) h = (long long)j1 - 1 + wl - q_offset + 1;
    if (h < l) h = l;
    *lo = (int)l;
    *hi = (int)h;
}
}  // namespace attn
