// paged_decode.cu -- paged MQA/GQA split-K decode attention for sm_103a.
//
// mainarch, decode-attention section: FlashDecoding-style split-KV online
// softmax, paged KV through a block table with a shuffled layout, GQA that
// reads each KV head once per group, FP8 KV dequantised in registers, and the
// memory-bound rules measured there (wide loads, many pages in flight before
// any cross-lane reduction, every buffer in device memory). Loom Kernels,
// "Attention" row: paged MQA/GQA decode with local split-K and LSE merge.
//
// Work decomposition. One CTA per (split s, kv head, sequence b) and four
// warps per CTA; the split's pages are dealt round-robin to the warps. Each
// warp runs its own ring of NSLOT page slots in shared memory: lane 0 issues
// TMA tile loads (cp.async.bulk.tensor, 128- or 64-byte swizzle) of the K and
// V rows of one page (16 tokens x D) into a slot and the slot's mbarrier
// completes when the bytes land; the warp consumes slot i while the next
// NSLOT-1 pages stream in, then refills the slot with page i + NSLOT. The
// block-table entries are read 32 at a time, one batch ahead, so the page
// id of every TMA issue is already in a register. Nothing waits across
// warps until the final combine.
//
// Math per page (16 tokens). The G <= 16 query heads of the group form the
// M = 16 rows of an mma.sync m16n8k16 tile (rows past G are zero), tokens
// are N, the head dim is K:
//   S[16 x 16] = Q[16 x D] . K^T      two n-tiles of 8 tokens, D/16 k-steps
//   online softmax on S in registers (each thread holds rows g and g+8,
//   token columns 2t, 2t+1; row max/sum need two quad shuffles)
//   O[16 x D] += P[16 x 16] . V        D/8 n-tiles, one k-step of 16 tokens
// bf16 caches feed ldmatrix (non-transposed for K, transposed for V) from
// the swizzled slots. E4M3 caches are loaded with 16-byte shared loads and
// converted to f16 in registers (cvt.rn.f16x2.e4m3x2, exact); the head-dim
// index is permuted consistently between Q and K so that each thread's
// bytes map straight onto its fragments, V's bytes are paired by token with
// prmt, and Q and P are f16. Scales fold into the score scale (k_scale) and
// the output (v_scale).
//
// NVFP4 caches (mainarch, decode-attention section: paged + GQA + 4-bit E2M1
// KV with block scales in one kernel; NVFP4 form) use the FP8 path's
// fragment mapping at half the bytes: a thread's 16-byte (K) or 8-byte (V)
// share of a row is one or two whole 16-value blocks, so each f16x2 word
// from cvt.rn.f16x2.e2m1x2 is multiplied (exactly) by its block's E4M3
// scale, loaded with the page by a 16-byte-aligned bulk copy beside the
// values. V pairs tokens by nibble: (a & 0x0F0F0F0F) | (b << 4 & 0xF0F0F0F0)
// puts value d of tokens a and b in one byte. Rows past the sequence end get
// a zero V scale (their nibbles are finite, so they contribute exactly 0).
//
// The tensor-core work is small (about 4*16*D flops per token and kv head
// against 4*D bytes of bf16 K/V): the kernel is bound by HBM, and mma.sync
// only keeps the ALU issue rate far from that bound. Scores and the softmax
// state are fp32; P enters the PV product as bf16 (bf16 caches) or f16 (FP8).
//
// Waits are bounded (about one second, then PKV_FLAG_WAIT_TIMEOUT is set,
// copies still in flight are waited for with the same bound, and the CTA
// finishes without hanging).
#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

// Launch shape: warps per CTA, shared-memory ring bytes per warp and the
// CTAs per SM the register budget is sized for (tuned on GB300; see the
// measurements recorded with the profiles).
#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 4
#endif
#ifndef PKV_DECODE_RING_BYTES
#define PKV_DECODE_RING_BYTES 16384
#endif
#ifndef PKV_DECODE_MIN_CTAS
#define PKV_DECODE_MIN_CTAS 3
#endif
constexpr int kWarps = PKV_DECODE_WARPS;
constexpr int kRingBytes = PKV_DECODE_RING_BYTES;
constexpr uint64_t kWaitLimitNs = 1000000000ull;

template <int D, int KIND>
struct Cfg {
    static constexpr bool F16 = KIND != kBf16;             // f16 mma operands (quantised caches)
    static constexpr int ROW = KIND == kBf16 ? 2 * D : (KIND == kFp8 ? D : D / 2);  // bytes of one token row
    static constexpr int E = KIND == kBf16 ? 2 : 1;        // bytes per tensor-map element
    static constexpr int BOXB = ROW >= 128 ? 128 : ROW;    // bytes per box row (swizzle span)
    static constexpr int NBOX = ROW / BOXB;                // boxes per page per tensor
    static constexpr int PAGE = kPageSize * ROW;           // bytes of one page of one head, K or V
    static constexpr int SROW = KIND == kFp4 ? D / 16 : 0; // block-scale bytes of one token row
    static constexpr int SPAGE = kPageSize * SROW;
    static constexpr int TX = 2 * PAGE + 2 * SPAGE;        // bytes landing per page
    // K, V, then the K and V block scales; a slot keeps the swizzle span's
    // alignment (8 rows of BOXB bytes)
    static constexpr int SLOT = (TX + 8 * BOXB - 1) / (8 * BOXB) * (8 * BOXB);
    static constexpr int NSLOT = kRingBytes / SLOT < 2 ? 2 : (kRingBytes / SLOT > 8 ? 8 : kRingBytes / SLOT);
    static constexpr int RING = NSLOT * SLOT;              // per warp
    // Pages consumed per iteration. Two (one softmax update per 32 tokens)
    // measured slower on GB300 for every ring size that fits: it halves the
    // pages a warp keeps in flight while it computes.
    static constexpr int PG = 1;
    static constexpr int KS = D / 16;                      // k-steps of QK
    static constexpr int NT = D / 8;                       // n-tiles of PV
    static constexpr int SMEM = kWarps * RING + kWarps * NSLOT * 8 + 1024;  // + barriers + alignment
    static_assert(BOXB == 128 || BOXB == 64 || BOXB == 32, "swizzle span");
    static_assert(RING >= (16 * (D + 8) + 32) * 4, "combine area must fit in a warp's ring");
};

// Byte offset of (row r, byte column col) in one page slice laid out by TMA
// with a 128-, 64- or 32-byte swizzle (the 16-byte chunk index is XOR-ed
// with address bits 7.. of the row start).
template <int BOXB>
__device__ __forceinline__ uint32_t swz(int r, int col) {
    if constexpr (BOXB == 128) {
        const int box = col >> 7;
        const int c = (col >> 4) & 7;
        return box * (kPageSize * 128) + r * 128 + ((c ^ (r & 7)) << 4) + (col & 15);
    } else if constexpr (BOXB == 64) {
        const int c = (col >> 4) & 3;
        return r * 64 + ((c ^ ((r >> 1) & 3)) << 4) + (col & 15);
    } else {
        const int c = (col >> 4) & 1;
        return r * 32 + ((c ^ ((r >> 2) & 1)) << 4) + (col & 15);
    }
}

__device__ __forceinline__ uint16_t lo16(uint32_t w) { return static_cast<uint16_t>(w & 0xFFFFu); }
__device__ __forceinline__ uint16_t hi16(uint32_t w) { return static_cast<uint16_t>(w >> 16); }

template <int D, int KIND, bool TWO>
__global__ void __launch_bounds__(kWarps * 32, PKV_DECODE_MIN_CTAS)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        const DecodeArgs a, const int hnd) {
    using C = Cfg<D, KIND>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem0 = smem_u32(smem);

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int s = blockIdx.x;
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;
    const int G = a.G;
    const int h0 = kvh * G;

    // ---- sequence bounds and this split's page range -----------------------
    // The block-table entries this warp needs first depend on the split's
    // first page, which depends on seq_len. They are read at the same time as
    // seq_len from the position a sequence of the full block-table width
    // would start at; the guess is kept when it turns out right (always, for
    // equal lengths) and re-read otherwise.
    const int pps_guess = (a.max_pages + a.num_splits - 1) / a.num_splits;
    const int p0_guess = s * pps_guess;
    const int32_t* bt_row = a.block_tables + b * a.bt_s0;
    auto guess_at = [&](int k) -> int {
        const int p = p0_guess + warp + kWarps * (k * 32 + lane);
        return p < a.max_pages ? __ldg(bt_row + p) : -1;
    };
    const int cur_guess = guess_at(0);
    const int nxt_guess = guess_at(1);
    int L = __ldg(a.seq_lens + b);
    const int cap = a.max_pages * kPageSize;
    if (L < 0 || L > cap) {
        if (threadIdx.x == 0 && s == 0 && kvh == 0) flag_error(a.err, PKV_FLAG_SEQ_LEN_RANGE);
        L = L < 0 ? 0 : cap;
    }
    const int npages = (L + kPageSize - 1) / kPageSize;
    const int pps = (npages + a.num_splits - 1) / a.num_splits;
    const int p0 = s * pps;
    const int p1 = min(p0 + pps, npages);
    float* outp = a.out_partial + b * a.op_s0 + s * a.op_s1 + h0 * a.op_s2;
    float* lsep = a.lse_partial + b * a.lp_s0 + s * a.lp_s1 + h0;
    if (p0 >= p1) {  // empty split: (0, -inf)
        grid_dep_wait();
        grid_dep_launch();
        for (int i = threadIdx.x; i < G * D; i += blockDim.x) outp[(i / D) * a.op_s2 + (i % D)] = 0.f;
        for (int i = threadIdx.x; i < G; i += blockDim.x) lsep[i] = -INFINITY;
        return;
    }
    const int npg = p1 - p0;
    const int nw = npg > warp ? (npg - warp + kWarps - 1) / kWarps : 0;  // this warp's pages

    uint8_t* ring = smem + warp * C::RING;
    const uint32_t ring0 = smem0 + warp * C::RING;
    const uint32_t bar0 = smem0 + kWarps * C::RING + warp * C::NSLOT * 8;

    if (lane == 0) {
        for (int i = 0; i < C::NSLOT; ++i) mbar_init(bar0 + 8 * i, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    __syncwarp();

    // ---- block-table batches (32 entries, one batch ahead) -----------------
    const int32_t* bt = bt_row + p0 + warp;
    auto load_batch = [&](int k) -> int {
        const int i = k * 32 + lane;
        return i < nw ? __ldg(bt + kWarps * i) : -1;
    };
    const bool guessed = p0 == p0_guess;
    int cur = guessed ? cur_guess : load_batch(0);
    int nxt = guessed ? nxt_guess : load_batch(1);
    const uint64_t policy = l2_policy_evict_first();
    const int64_t num_pages = a.num_pages;
    float ks = 1.f, vs = 1.f;
    if constexpr (KIND != kBf16) {
        ks = __ldg(a.k_scale + (a.n_scale == 1 ? 0 : kvh));
        vs = __ldg(a.v_scale + (a.n_scale == 1 ? 0 : kvh));
    }

    // Everything above reads only this call's index inputs. q and the cache
    // may still be being written by the preceding cache-write grid (launched
    // as our programmatic predecessor): wait for it before touching them.
    grid_dep_wait();
    grid_dep_launch();

    auto page_id = [&](int i, int cur_batch) -> int {
        const int src = ((i >> 5) == cur_batch) ? cur : nxt;
        return __shfl_sync(0xffffffffu, src, i & 31);
    };
    auto issue = [&](int i, int pid) {  // called by lane 0
        const int slot = i % C::NSLOT;
        const uint32_t bar = bar0 + 8 * slot;
        if (pid < 0 || pid >= num_pages) {
            mbar_arrive(bar);  // completes the phase with no bytes; the page is skipped
            return;
        }
        mbar_arrive_expect_tx(bar, C::TX);
        const uint32_t kdst = ring0 + slot * C::SLOT;
        const uint32_t vdst = kdst + C::PAGE;
        const int c1 = hnd ? 0 : kvh;
        const int c2 = hnd ? kvh : 0;
#pragma unroll
        for (int bx = 0; bx < C::NBOX; ++bx) {
            const int d0 = bx * (C::BOXB / C::E);
            tma_load_4d(kdst + bx * kPageSize * C::BOXB, &tmk, bar, d0, c1, c2, pid, policy);
            tma_load_4d(vdst + bx * kPageSize * C::BOXB, &tmv, bar, d0, c1, c2, pid, policy);
        }
        if constexpr (KIND == kFp4) {
            bulk_load(kdst + 2 * C::PAGE, a.k_bs + pid * a.kbs_s0 + kvh * a.kbs_s1, C::SPAGE, bar, policy);
            bulk_load(kdst + 2 * C::PAGE + C::SPAGE, a.v_bs + pid * a.vbs_s0 + kvh * a.vbs_s1, C::SPAGE, bar,
                      policy);
        }
    };

    // prologue: fill the ring
    {
        const int n0 = min(C::NSLOT, nw);
        for (int i = 0; i < n0; ++i) {
            const int pid = page_id(i, 0);
            if (lane == 0) issue(i, pid);
        }
    }

    // ---- Q fragments (A operand), loaded once -------------------------------
    uint32_t qa[C::KS][4];
    {
        const uint16_t* qb = a.q + b * a.q_s0 + h0 * a.q_s1;
        const bool rg = g < G;
        const bool rg8 = TWO && (g + 8 < G);
#pragma unroll
        for (int j = 0; j < C::KS; ++j) {
            int dlo, dhi;
            if constexpr (C::F16) {
                dlo = (D / 4) * t + 4 * j;
                dhi = dlo + 2;
            } else {
                dlo = 16 * j + 2 * t;
                dhi = dlo + 8;
            }
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            if (rg) {
                w[0] = __ldg(reinterpret_cast<const uint32_t*>(qb + g * a.q_s1 + dlo));
                w[2] = __ldg(reinterpret_cast<const uint32_t*>(qb + g * a.q_s1 + dhi));
            }
            if (rg8) {
                w[1] = __ldg(reinterpret_cast<const uint32_t*>(qb + (g + 8) * a.q_s1 + dlo));
                w[3] = __ldg(reinterpret_cast<const uint32_t*>(qb + (g + 8) * a.q_s1 + dhi));
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if constexpr (C::F16)
                    qa[j][e] = pack_f16(bf16_lo(w[e]), bf16_hi(w[e]));
                else
                    qa[j][e] = w[e];
            }
        }
    }

    const float sl = a.scale_log2 * ks;

    float acc[C::NT][4];
#pragma unroll
    for (int n = 0; n < C::NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    bool ok = true;
    int bad_pages = 0;
    int i = 0;

    // S = Q K^T for the 16 tokens of the page at kb: sc[nt] holds tokens
    // 8nt + 2t, 8nt + 2t + 1 of rows g and g + 8.
    auto qk_page = [&](uint32_t kb, float (*sc)[4]) {
        if constexpr (KIND == kBf16) {
#pragma unroll
            for (int jj = 0; jj < C::KS / 2; ++jj) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int r = 8 * nt + (lane & 7);
                    const int col = 2 * (32 * jj + 8 * (lane >> 3));
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kb + swz<C::BOXB>(r, col), b0, b1, b2, b3);
                    mma16816<false>(sc[nt], qa[2 * jj][0], qa[2 * jj][1], qa[2 * jj][2], qa[2 * jj][3], b0, b1);
                    mma16816<false>(sc[nt], qa[2 * jj + 1][0], qa[2 * jj + 1][1], qa[2 * jj + 1][2],
                                    qa[2 * jj + 1][3], b2, b3);
                }
            }
        } else if constexpr (KIND == kFp4) {
            // thread t's share of row r: bytes [ (D/8)t, (D/8)(t+1) ), i.e.
            // values [(D/4)t, (D/4)(t+1)) -- blocks 2t, 2t+1 (D = 128) or t
            const uint32_t kbs = kb + 2 * C::PAGE;  // K block scales [16][D/16]
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int r = 8 * nt + g;
                constexpr int NW = D / 32;          // words of E2M1 pairs per thread
                uint32_t w[NW];
                uint32_t sA, sB;                    // {s, s} of the first / second block
                if constexpr (D == 128) {
                    const uint4 x0 = lds128(kb + swz<C::BOXB>(r, 16 * t));
                    w[0] = x0.x; w[1] = x0.y; w[2] = x0.z; w[3] = x0.w;
                    const uint32_t s2 = e4m3x2_to_f16x2(static_cast<uint16_t>(lds16(kbs + r * C::SROW + 2 * t)));
                    sA = prmt(s2, s2, 0x1010u);
                    sB = prmt(s2, s2, 0x3232u);
                } else {
                    const uint2 x0 = lds64(kb + swz<C::BOXB>(r, 8 * t));
                    w[0] = x0.x; w[1] = x0.y;
                    const uint32_t s1 = lds8(kbs + r * C::SROW + t);
                    sA = sB = e4m3x2_to_f16x2(static_cast<uint16_t>(s1 | (s1 << 8)));
                }
#pragma unroll
                for (int wi = 0; wi < NW; ++wi) {
                    uint32_t h[4];
                    e2m1x8_to_f16x2(w[wi], h);
                    const uint32_t sc2 = (D == 128 && wi >= 2) ? sB : sA;
#pragma unroll
                    for (int e = 0; e < 4; ++e) h[e] = hmul2(h[e], sc2);
                    const int j = 2 * wi;
                    mma16816<true>(sc[nt], qa[j][0], qa[j][1], qa[j][2], qa[j][3], h[0], h[1]);
                    mma16816<true>(sc[nt], qa[j + 1][0], qa[j + 1][1], qa[j + 1][2], qa[j + 1][3], h[2], h[3]);
                }
            }
        } else {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int r = 8 * nt + g;
                uint32_t w[C::KS];
                if constexpr (D == 128) {
                    const uint4 x0 = lds128(kb + swz<C::BOXB>(r, 32 * t));
                    const uint4 x1 = lds128(kb + swz<C::BOXB>(r, 32 * t + 16));
                    w[0] = x0.x; w[1] = x0.y; w[2] = x0.z; w[3] = x0.w;
                    w[4] = x1.x; w[5] = x1.y; w[6] = x1.z; w[7] = x1.w;
                } else {
                    const uint4 x0 = lds128(kb + swz<C::BOXB>(r, 16 * t));
                    w[0] = x0.x; w[1] = x0.y; w[2] = x0.z; w[3] = x0.w;
                }
#pragma unroll
                for (int j = 0; j < C::KS; ++j)
                    mma16816<true>(sc[nt], qa[j][0], qa[j][1], qa[j][2], qa[j][3], e4m3x2_to_f16x2(lo16(w[j])),
                                   e4m3x2_to_f16x2(hi16(w[j])));
            }
        }
    };
    // O += P V for the page at vb; tokens at or past `valid` contribute zero
    // (their V bytes may be anything, so they are zeroed, not only weighted 0).
    auto pv_page = [&](uint32_t vb, int valid, uint32_t pa0, uint32_t pa1, uint32_t pa2, uint32_t pa3) {
        if constexpr (KIND == kBf16) {
            uint32_t mk0 = 0xFFFFFFFFu, mk1 = 0xFFFFFFFFu;
            if (valid < kPageSize) {
                mk0 = (2 * t < valid ? 0x0000FFFFu : 0u) | (2 * t + 1 < valid ? 0xFFFF0000u : 0u);
                mk1 = (2 * t + 8 < valid ? 0x0000FFFFu : 0u) | (2 * t + 9 < valid ? 0xFFFF0000u : 0u);
            }
#pragma unroll
            for (int dp = 0; dp < C::NT / 2; ++dp) {
                const int mi = lane >> 3;
                const int r = 8 * (mi & 1) + (lane & 7);
                const int col = 16 * (2 * dp + (mi >> 1));
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vb + swz<C::BOXB>(r, col), b0, b1, b2, b3);
                mma16816<false>(acc[2 * dp], pa0, pa1, pa2, pa3, b0 & mk0, b1 & mk1);
                mma16816<false>(acc[2 * dp + 1], pa0, pa1, pa2, pa3, b2 & mk0, b3 & mk1);
            }
        } else if constexpr (KIND == kFp4) {
            // thread g's share of each row: bytes [(D/16)g, (D/16)(g+1)), values
            // d = (D/8)g + jn, jn < D/8 -- all in block g (D = 128) or g/2
            constexpr int NWD = D / 64;  // words of E2M1 pairs per token row per thread
            const uint32_t vbs = vb + C::PAGE + C::SPAGE;  // V block scales [16][D/16]
            const int blk = D == 128 ? g : (g >> 1);
            uint32_t va[4][NWD];
            uint32_t sb4 = 0u;  // scale bytes of rows 2t, 2t+1, 2t+8, 2t+9
            const int rows[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if constexpr (D == 128) {
                    const uint2 xv = lds64(vb + swz<C::BOXB>(rows[q], 8 * g));
                    va[q][0] = xv.x; va[q][1] = xv.y;
                } else {
                    va[q][0] = lds32(vb + swz<C::BOXB>(rows[q], 4 * g));
                }
                const uint32_t sbq = lds8(vbs + rows[q] * C::SROW + blk);
                sb4 |= (rows[q] < valid ? sbq : 0u) << (8 * q);
            }
            const uint32_t s01 = e4m3x2_to_f16x2(lo16(sb4));  // {s(2t), s(2t+1)}
            const uint32_t s89 = e4m3x2_to_f16x2(hi16(sb4));  // {s(2t+8), s(2t+9)}
#pragma unroll
            for (int wd = 0; wd < NWD; ++wd) {
                // byte i of xe: value 2i of tokens 2t (low nibble) and 2t+1;
                // xo: value 2i+1; ye / yo the same for tokens 2t+8, 2t+9
                const uint32_t xe = (va[0][wd] & 0x0F0F0F0Fu) | ((va[1][wd] << 4) & 0xF0F0F0F0u);
                const uint32_t xo = ((va[0][wd] >> 4) & 0x0F0F0F0Fu) | (va[1][wd] & 0xF0F0F0F0u);
                const uint32_t ye = (va[2][wd] & 0x0F0F0F0Fu) | ((va[3][wd] << 4) & 0xF0F0F0F0u);
                const uint32_t yo = ((va[2][wd] >> 4) & 0x0F0F0F0Fu) | (va[3][wd] & 0xF0F0F0F0u);
                uint32_t he[4], ho[4], ge[4], go[4];
                e2m1x8_to_f16x2(xe, he);
                e2m1x8_to_f16x2(xo, ho);
                e2m1x8_to_f16x2(ye, ge);
                e2m1x8_to_f16x2(yo, go);
#pragma unroll
                for (int i2 = 0; i2 < 4; ++i2) {
                    const int jn = 8 * wd + 2 * i2;
                    mma16816<true>(acc[jn], pa0, pa1, pa2, pa3, hmul2(he[i2], s01), hmul2(ge[i2], s89));
                    mma16816<true>(acc[jn + 1], pa0, pa1, pa2, pa3, hmul2(ho[i2], s01), hmul2(go[i2], s89));
                }
            }
        } else {
            constexpr int NWD = D / 32;  // words of V bytes per token row per thread
            uint32_t va[4][NWD];
            const int rows[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if constexpr (D == 128) {
                    const uint4 xv = lds128(vb + swz<C::BOXB>(rows[q], 16 * g));
                    va[q][0] = xv.x; va[q][1] = xv.y; va[q][2] = xv.z; va[q][3] = xv.w;
                } else {
                    const uint2 xv = lds64(vb + swz<C::BOXB>(rows[q], 8 * g));
                    va[q][0] = xv.x; va[q][1] = xv.y;
                }
                if (rows[q] >= valid) {
#pragma unroll
                    for (int wd = 0; wd < NWD; ++wd) va[q][wd] = 0u;
                }
            }
#pragma unroll
            for (int wd = 0; wd < NWD; ++wd) {
                const uint32_t pl = prmt(va[0][wd], va[1][wd], 0x5140u);
                const uint32_t ph = prmt(va[0][wd], va[1][wd], 0x7362u);
                const uint32_t ql = prmt(va[2][wd], va[3][wd], 0x5140u);
                const uint32_t qh = prmt(va[2][wd], va[3][wd], 0x7362u);
                mma16816<true>(acc[4 * wd + 0], pa0, pa1, pa2, pa3, e4m3x2_to_f16x2(lo16(pl)),
                               e4m3x2_to_f16x2(lo16(ql)));
                mma16816<true>(acc[4 * wd + 1], pa0, pa1, pa2, pa3, e4m3x2_to_f16x2(hi16(pl)),
                               e4m3x2_to_f16x2(hi16(ql)));
                mma16816<true>(acc[4 * wd + 2], pa0, pa1, pa2, pa3, e4m3x2_to_f16x2(lo16(ph)),
                               e4m3x2_to_f16x2(lo16(qh)));
                mma16816<true>(acc[4 * wd + 3], pa0, pa1, pa2, pa3, e4m3x2_to_f16x2(hi16(ph)),
                               e4m3x2_to_f16x2(hi16(qh)));
            }
        }
    };

    // Pages are consumed PG at a time; one softmax update covers all their
    // tokens.
    constexpr int PG = C::PG;
    for (; i < nw; i += PG) {
        if (i > 0 && (i & 31) == 0) {
            cur = nxt;
            nxt = load_batch((i >> 5) + 1);
        }
        bool landed = true;
#pragma unroll
        for (int j = 0; j < PG; ++j) {
            const int ij = i + j;
            if (ij < nw) landed &= mbar_wait_bounded(bar0 + 8 * (ij % C::NSLOT), (ij / C::NSLOT) & 1, kWaitLimitNs);
        }
        if (!__all_sync(0xffffffffu, landed)) {
            ok = false;
            break;
        }
        int valid[PG];
        bool any = false;
#pragma unroll
        for (int j = 0; j < PG; ++j) {
            const int ij = i + j;
            const int pid = page_id(ij, i >> 5);
            const bool pid_ok = pid >= 0 && pid < num_pages;
            if (ij < nw && !pid_ok) ++bad_pages;
            const int p = p0 + warp + kWarps * ij;
            valid[j] = (ij < nw && pid_ok) ? min(kPageSize, L - p * kPageSize) : 0;
            any |= valid[j] > 0;
        }
        if (any) {
            float sc[2 * PG][4];
#pragma unroll
            for (int n = 0; n < 2 * PG; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
            for (int j = 0; j < PG; ++j)
                if (valid[j] > 0) qk_page(ring0 + ((i + j) % C::NSLOT) * C::SLOT, &sc[2 * j]);

            // ---- online softmax (log2 domain) -------------------------------
            float x[2 * PG][4];
#pragma unroll
            for (int n = 0; n < 2 * PG; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = 8 * (n & 1) + 2 * t + (e & 1);
                    x[n][e] = tok < valid[n >> 1] ? sc[n][e] * sl : -INFINITY;
                }
            float pmA = -INFINITY, pmB = -INFINITY;
#pragma unroll
            for (int n = 0; n < 2 * PG; ++n) {
                pmA = fmaxf(pmA, fmaxf(x[n][0], x[n][1]));
                if constexpr (TWO) pmB = fmaxf(pmB, fmaxf(x[n][2], x[n][3]));
            }
            pmA = fmaxf(pmA, __shfl_xor_sync(0xffffffffu, pmA, 1));
            pmA = fmaxf(pmA, __shfl_xor_sync(0xffffffffu, pmA, 2));
            const float nA = fmaxf(mA, pmA);
            const float alA = fast_exp2(mA - nA);
            mA = nA;
            float nB = 0.f, alB = 1.f;
            if constexpr (TWO) {
                pmB = fmaxf(pmB, __shfl_xor_sync(0xffffffffu, pmB, 1));
                pmB = fmaxf(pmB, __shfl_xor_sync(0xffffffffu, pmB, 2));
                nB = fmaxf(mB, pmB);
                alB = fast_exp2(mB - nB);
                mB = nB;
            }
            float pr[2 * PG][4];
            float sA = 0.f, sB = 0.f;
#pragma unroll
            for (int n = 0; n < 2 * PG; ++n) {
                pr[n][0] = fast_exp2(x[n][0] - nA);
                pr[n][1] = fast_exp2(x[n][1] - nA);
                sA += pr[n][0] + pr[n][1];
                if constexpr (TWO) {
                    pr[n][2] = fast_exp2(x[n][2] - nB);
                    pr[n][3] = fast_exp2(x[n][3] - nB);
                    sB += pr[n][2] + pr[n][3];
                } else {
                    pr[n][2] = pr[n][3] = 0.f;
                }
            }
            lA = lA * alA + sA;
            if constexpr (TWO) lB = lB * alB + sB;
            // rescale the accumulators only when some row's max moved (after
            // the first pages it rarely does)
            if (__any_sync(0xffffffffu, alA != 1.f || alB != 1.f)) {
#pragma unroll
                for (int n = 0; n < C::NT; ++n) {
                    acc[n][0] *= alA;
                    acc[n][1] *= alA;
                    if constexpr (TWO) {
                        acc[n][2] *= alB;
                        acc[n][3] *= alB;
                    }
                }
            }
            // ---- O += P V, page by page (P as the A operand: rows g / g+8,
            // tokens 2t.. and 8+2t.. of the page) -----------------------------
#pragma unroll
            for (int j = 0; j < PG; ++j) {
                if (valid[j] <= 0) continue;
                const float* p0r = pr[2 * j];
                const float* p1r = pr[2 * j + 1];
                uint32_t pa0, pa1 = 0u, pa2, pa3 = 0u;
                if constexpr (C::F16) {
                    pa0 = pack_f16(p0r[0], p0r[1]);
                    pa2 = pack_f16(p1r[0], p1r[1]);
                    if constexpr (TWO) {
                        pa1 = pack_f16(p0r[2], p0r[3]);
                        pa3 = pack_f16(p1r[2], p1r[3]);
                    }
                } else {
                    pa0 = pack_bf16(p0r[0], p0r[1]);
                    pa2 = pack_bf16(p1r[0], p1r[1]);
                    if constexpr (TWO) {
                        pa1 = pack_bf16(p0r[2], p0r[3]);
                        pa3 = pack_bf16(p1r[2], p1r[3]);
                    }
                }
                pv_page(ring0 + ((i + j) % C::NSLOT) * C::SLOT + C::PAGE, valid[j], pa0, pa1, pa2, pa3);
            }
        }

        // ---- refill the consumed slots with pages i + NSLOT .. ----------------
        __syncwarp();
#pragma unroll
        for (int j = 0; j < PG; ++j) {
            const int nx = i + j + C::NSLOT;
            if (nx < nw) {
                const int pid2 = page_id(nx, i >> 5);
                if (lane == 0) {
                    fence_proxy_async_smem();
                    issue(nx, pid2);
                }
            }
        }
    }

    if (!ok) {
        // A copy never landed: record it, then wait (bounded) for every copy
        // still in flight before the shared memory is reused or released.
        if (lane == 0) flag_error(a.err, PKV_FLAG_WAIT_TIMEOUT);
        const int last = min(i + C::NSLOT, nw);
        for (int j = i; j < last; ++j)
            (void)mbar_wait_bounded(bar0 + 8 * (j % C::NSLOT), (j / C::NSLOT) & 1, kWaitLimitNs);
    }
    if (bad_pages && lane == 0) flag_error(a.err, PKV_FLAG_PAGE_RANGE);

    // ---- per-warp state -> shared memory (the warp's own ring) ----------------
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    if constexpr (TWO) {
        lB += __shfl_xor_sync(0xffffffffu, lB, 1);
        lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    }
    __syncwarp();
    // [16][D + 8] partial sums (the 8-float pad makes the float2 stores of
    // the eight row groups fall on distinct banks), then m[16], l[16]
    constexpr int CWS = D + 8;
    float* cw = reinterpret_cast<float*>(ring);
    float* cm = cw + 16 * CWS;
    float* cl = cm + 16;
    if (t == 0) {
        cm[g] = mA;
        cl[g] = lA;
        cm[g + 8] = TWO ? mB : -INFINITY;
        cl[g + 8] = TWO ? lB : 0.f;
    }
#pragma unroll
    for (int n = 0; n < C::NT; ++n) {
        if constexpr (C::F16) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int d = (D / 8) * (2 * t + e) + n;
                cw[g * CWS + d] = acc[n][e];
                if constexpr (TWO) cw[(g + 8) * CWS + d] = acc[n][2 + e];
            }
        } else {
            const int d = 8 * n + 2 * t;
            *reinterpret_cast<float2*>(cw + g * CWS + d) = make_float2(acc[n][0], acc[n][1]);
            if constexpr (TWO) *reinterpret_cast<float2*>(cw + (g + 8) * CWS + d) = make_float2(acc[n][2], acc[n][3]);
        }
    }
    __syncthreads();

    // ---- combine the four warps ------------------------------------------------
    __shared__ float wgt[kWarps][16];
    __shared__ float inv_l[16];
    if (threadIdx.x < G) {
        const int r = threadIdx.x;
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) {
            const float* cmw = reinterpret_cast<const float*>(smem + w * C::RING) + 16 * CWS;
            M = fmaxf(M, cmw[r]);
        }
        float Lsum = 0.f;
        for (int w = 0; w < kWarps; ++w) {
            const float* cmw = reinterpret_cast<const float*>(smem + w * C::RING) + 16 * CWS;
            const float ww = (M == -INFINITY || cmw[r] == -INFINITY) ? 0.f : exp2f(cmw[r] - M);
            wgt[w][r] = ww;
            Lsum += ww * cmw[16 + r];
        }
        const bool empty = !(Lsum > 0.f);
        inv_l[r] = empty ? 0.f : vs / Lsum;
        lsep[r] = empty ? -INFINITY : (M + __log2f(Lsum)) * 0.69314718055994530942f;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int r = idx / D;
        const int d = idx - r * D;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) o += wgt[w][r] * reinterpret_cast<const float*>(smem + w * C::RING)[r * CWS + d];
        outp[r * a.op_s2 + d] = o * inv_l[r];
    }
}

template <int D, int KIND, bool TWO>
cudaError_t launch_t(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int hnd, cudaStream_t s) {
    using C = Cfg<D, KIND>;
    auto kern = paged_decode_kernel<D, KIND, TWO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid(a.num_splits, a.Hkv, a.B);
    return launch_dependent(kern, grid, dim3(kWarps * 32), C::SMEM, s, tk, tv, a, hnd);
}

template <int D, int KIND>
cudaError_t launch_g(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int hnd, cudaStream_t s) {
    return a.G > 8 ? launch_t<D, KIND, true>(a, tk, tv, hnd, s) : launch_t<D, KIND, false>(a, tk, tv, hnd, s);
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int hnd, cudaStream_t s) {
    switch (a.kind) {
        case kBf16: return launch_g<D, kBf16>(a, tk, tv, hnd, s);
        case kFp8: return launch_g<D, kFp8>(a, tk, tv, hnd, s);
        case kFp4: return launch_g<D, kFp4>(a, tk, tv, hnd, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int decode_ctas_per_sm(int D, int kind) {
    (void)D;
    (void)kind;
    return PKV_DECODE_MIN_CTAS;
}

cudaError_t launch_paged_decode(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    const int hnd = a.layout == PKV_HND;
    if (a.D == 128) return launch_d<128>(a, tk, tv, hnd, s);
    if (a.D == 64) return launch_d<64>(a, tk, tv, hnd, s);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
