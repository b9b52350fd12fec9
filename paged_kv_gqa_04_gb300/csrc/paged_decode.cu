// paged_decode.cu -- paged MQA/GQA split-K decode attention for sm_103a.
//
// mainarch, decode-attention section: FlashDecoding-style split-KV online
// softmax, paged KV through a block table with a shuffled layout, GQA that
// reads each KV head once per group, FP8 and 4-bit KV dequantised in
// registers, and the memory-bound rules measured there (wide loads, many
// pages in flight before any cross-lane reduction, every buffer in device
// memory). Loom Kernels, "Attention" row: paged MQA/GQA decode with local
// split-K and LSE merge.
//
// Work decomposition. One CTA per (split s, kv head, sequence b) and four
// warps per CTA; the split's pages are dealt round-robin to the warps. Each
// warp runs its own ring of NSLOT page slots in shared memory: its lanes
// issue TMA tile loads (cp.async.bulk.tensor, 128-, 64- or 32-byte swizzle)
// of the K and V rows of one page (16 tokens x D) into a slot, one copy per
// lane, and the slot's mbarrier completes when the bytes land; the warp
// consumes slot i while the next NSLOT-1 pages stream in, then refills the
// slot with page i + NSLOT.
// The block-table entries are read 32 at a time, one batch ahead, so the
// page id of every TMA issue is already in a register. Nothing waits across
// warps until the final combine.
//
// Math per page (16 tokens), with the cache on the M side of mma.sync
// m16n8k16 and the query heads of the group on N (8 heads per n-tile, one
// tile for G <= 8, two for G <= 16; heads past G are zero):
//   S^T[16 tok x 8 h] = K[16 x D] . Q^T      D/16 k-steps
//   online softmax on S^T in registers: a thread holds tokens g, g+8 of
//   heads 2t, 2t+1; a head's max over the page is three xor-shuffles over
//   the eight lanes g
//   P^T as the B operand: the f16/bf16-packed S^T fragment of each 8-token
//   half, transposed in registers with movmatrix (bf16: two terms, the
//   rounded weight and its rounded rest, each multiplied by V^T)
//   O^T[16 d x 8 h] += V^T[16 x 16 tok] . P^T    D/16 m-tiles
// With the cache as the A operand one mma covers 16 tokens (K) or 16
// head-dim values (V) of all the group's heads: half the mma count of the
// heads-as-M form for G <= 8, and half its accumulator and Q registers.
//
// bf16 caches feed ldmatrix (non-transposed for K, transposed for V) from
// the swizzled slots. Quantised caches are loaded with 16/8-byte shared
// loads and converted to f16 in registers: E4M3 with cvt.rn.f16x2.e4m3x2,
// E2M1 with cvt.rn.f16x2.e2m1x2 followed by an f16x2 multiply by the block's
// E4M3 scale (both exact). The head-dim index is permuted consistently
// between Q and K so that each thread's bytes map straight onto its
// fragments (thread t holds head-dim values [D/4 t, D/4 (t+1)) of K rows g
// and g+8); V's bytes are paired by token, with prmt (E4M3) or a nibble
// interleave (a & 0x0F0F0F0F) | (b << 4 & 0xF0F0F0F0) (E2M1), and thread g
// owns head-dim values [D/8 g, D/8 (g+1)) of V. Q and P are then f16.
// Static scales fold into the score scale (k_scale) and the output
// (v_scale). NVFP4 block scales land with the page by a 16-byte-aligned
// bulk copy beside the values (HND only); rows past the sequence end get a
// zero V scale (their nibbles are finite, so they contribute exactly 0).
//
// The tensor-core work is small (about 4*16*D flops per token and kv head
// against 4*D bytes of bf16 K/V): the kernel is bound by HBM for bf16, and
// by the dequantisation's ALU issue for the 1- and 1/2-byte formats, which
// is why the register budget is sized for four CTAs per SM there. Scores
// and the softmax state are fp32.
//
// Waits are bounded (about one second, then PKV_FLAG_WAIT_TIMEOUT is set,
// copies still in flight are waited for with the same bound, and the CTA
// finishes without hanging).
#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

// Launch shape per cache format: shared-memory ring bytes per warp and the
// CTAs per SM that registers and shared memory are sized for (tuned on
// GB300; see the measurements recorded with the profiles).
#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 4
#endif
#ifndef PKV_DECODE_RING_BF16
#define PKV_DECODE_RING_BF16 16384
#endif
#ifndef PKV_DECODE_CTAS_BF16
#define PKV_DECODE_CTAS_BF16 3
#endif
#ifndef PKV_DECODE_RING_FP8
#define PKV_DECODE_RING_FP8 12288
#endif
#ifndef PKV_DECODE_CTAS_FP8
#define PKV_DECODE_CTAS_FP8 4
#endif
#ifndef PKV_DECODE_RING_FP4
#define PKV_DECODE_RING_FP4 12800
#endif
#ifndef PKV_DECODE_CTAS_FP4
#define PKV_DECODE_CTAS_FP4 4
#endif
constexpr int kWarps = PKV_DECODE_WARPS;
constexpr uint64_t kWaitLimitNs = 1000000000ull;

constexpr int ring_bytes(int kind) {
    return kind == kBf16 ? PKV_DECODE_RING_BF16 : (kind == kFp8 ? PKV_DECODE_RING_FP8 : PKV_DECODE_RING_FP4);
}
// Two head tiles (G > 8) need twice the accumulators: at most three CTAs.
constexpr int ctas_per_sm(int kind, int nh) {
    const int c = kind == kBf16 ? PKV_DECODE_CTAS_BF16 : (kind == kFp8 ? PKV_DECODE_CTAS_FP8 : PKV_DECODE_CTAS_FP4);
    return nh == 2 && c > 3 ? 3 : c;
}

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
    static constexpr int RB = ring_bytes(KIND);
    static constexpr int NSLOT = RB / SLOT < 2 ? 2 : (RB / SLOT > 8 ? 8 : RB / SLOT);
    static constexpr int RING = NSLOT * SLOT;              // per warp
    static constexpr int KS = D / 16;                      // k-steps of K.Q^T = m-tiles of V^T.P^T
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

template <int D, int KIND, int NH>
__global__ void __launch_bounds__(kWarps * 32, ctas_per_sm(KIND, NH))
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
    // ---- which split of which sequence ----------------------------------------
    // Uniform launch: split blockIdx.x of kv head blockIdx.y of sequence
    // blockIdx.z, every sequence in num_splits splits. Planned launch (a
    // 1-D grid): CTA x takes kv head x % Hkv of work item x / Hkv, so the
    // hardware dispatches the items in the plan's order (longest first) with
    // all kv heads of an item together; the item names the sequence and the
    // split, and the sequence's own split count comes from splits_per_seq
    // (clamped to [1, num_splits], the records there are).
    int b, s, kvh, p0_guess;
    if (a.work == nullptr) {
        s = blockIdx.x;
        kvh = blockIdx.y;
        b = blockIdx.z;
        p0_guess = s * ((a.max_pages + a.num_splits - 1) / a.num_splits);
    } else {
        const int item = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.Hkv));
        kvh = static_cast<int>(blockIdx.x - static_cast<unsigned>(item) * a.Hkv);
        const int2 e = __ldg(reinterpret_cast<const int2*>(a.work) + item);
        b = e.x >> 12;
        s = e.x & 0xFFF;
        p0_guess = min(max(e.y, -1), a.max_pages);  // a hint only: kept in range, checked below
        if (b < 0 || b >= a.B || s >= a.num_splits) {  // an entry outside the batch or the records
            if (threadIdx.x == 0 && kvh == 0) flag_error(a.err, PKV_FLAG_PLAN_RANGE);
            grid_dep_wait();
            grid_dep_launch();
            return;
        }
    }
    const int G = a.G;
    const int h0 = kvh * G;

    // ---- sequence bounds and this split's page range -----------------------
    // The block-table entries this warp needs first depend on the split's
    // first page, which depends on seq_len. They are read at the same time as
    // seq_len from a guessed first page -- where a sequence of the full
    // block-table width would start (uniform), or the plan's first page
    // (planned); the guess is kept when it turns out right (always, for
    // equal lengths or a plan made from these lengths) and re-read otherwise.
    const int32_t* bt_row = a.block_tables + b * a.bt_s0;
    auto guess_at = [&](int k) -> int {
        const int p = p0_guess + warp + kWarps * (k * 32 + lane);
        return (p >= 0 && p < a.max_pages) ? __ldg(bt_row + p) : -1;  // a plan's hint may be anything
    };
    const int cur_guess = guess_at(0);
    const int nxt_guess = guess_at(1);
    int L = __ldg(a.seq_lens + b);
    int S_b = a.num_splits;
    if (a.splits_per_seq != nullptr) {
        const int r = __ldg(a.splits_per_seq + b);
        S_b = min(max(r, 1), a.num_splits);
        if ((r != S_b || s >= S_b) && threadIdx.x == 0 && kvh == 0) flag_error(a.err, PKV_FLAG_PLAN_RANGE);
    }
    const int cap = a.max_pages * kPageSize;
    if (L < 0 || L > cap) {
        if (threadIdx.x == 0 && s == 0 && kvh == 0) flag_error(a.err, PKV_FLAG_SEQ_LEN_RANGE);
        L = L < 0 ? 0 : cap;
    }
    const int npages = (L + kPageSize - 1) / kPageSize;
    const int pps = (npages + S_b - 1) / S_b;
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
    // Start the copies of page `pid` into ring slot `slot`; called by the
    // whole warp (pid is warp-uniform). Lane 0 posts the byte count, then
    // each copy is issued by its own lane: lane 2 bx + v copies box bx of K
    // (v = 0) or V (v = 1); NVFP4 scales come from the next two lanes.
    constexpr int NCOPY = 2 * C::NBOX + (KIND == kFp4 ? 2 : 0);
    auto issue = [&](int slot, int pid) {
        const uint32_t bar = bar0 + 8 * slot;
        if (pid < 0 || pid >= num_pages) {
            if (lane == 0) mbar_arrive(bar);  // completes the phase with no bytes; the page is skipped
            return;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar, C::TX);
        __syncwarp();
        const uint32_t kdst = ring0 + slot * C::SLOT;
        const int v = lane & 1;
        if (lane < 2 * C::NBOX) {
            const int bx = lane >> 1;
            tma_load_4d(kdst + v * C::PAGE + bx * kPageSize * C::BOXB, v ? &tmv : &tmk, bar, bx * (C::BOXB / C::E),
                        hnd ? 0 : kvh, hnd ? kvh : 0, pid, policy);
        } else if (KIND == kFp4 && lane < NCOPY) {
            const uint8_t* src = v ? a.v_bs + pid * a.vbs_s0 + kvh * a.vbs_s1 : a.k_bs + pid * a.kbs_s0 + kvh * a.kbs_s1;
            bulk_load(kdst + 2 * C::PAGE + v * C::SPAGE, src, C::SPAGE, bar, policy);
        }
    };

    // prologue: fill the ring
    {
        const int n0 = min(C::NSLOT, nw);
        for (int i = 0; i < n0; ++i) issue(i, page_id(i, 0));
    }

    // ---- Q^T fragments (B operand), loaded once: head 8 ht + g ------------
    // k-step kk, k-rows 2t, 2t+1 (b0) and 2t+8, 2t+9 (b1) are head-dim values
    // 16 kk + 2t (+8) for bf16, and (D/4) t + 4 kk (+2) for the quantised
    // formats (the order in which a thread's cache bytes hold them).
    uint32_t qb[NH][C::KS][2];
    {
        const uint16_t* qbase = a.q + b * a.q_s0 + h0 * a.q_s1;
#pragma unroll
        for (int ht = 0; ht < NH; ++ht) {
            const int h = 8 * ht + g;
            const bool live = h < G;
#pragma unroll
            for (int kk = 0; kk < C::KS; ++kk) {
                const int dlo = C::F16 ? (D / 4) * t + 4 * kk : 16 * kk + 2 * t;
                const int dhi = C::F16 ? dlo + 2 : dlo + 8;
                uint32_t w0 = 0u, w1 = 0u;
                if (live) {
                    w0 = __ldg(reinterpret_cast<const uint32_t*>(qbase + h * a.q_s1 + dlo));
                    w1 = __ldg(reinterpret_cast<const uint32_t*>(qbase + h * a.q_s1 + dhi));
                }
                if constexpr (C::F16) {
                    qb[ht][kk][0] = pack_f16(bf16_lo(w0), bf16_hi(w0));
                    qb[ht][kk][1] = pack_f16(bf16_lo(w1), bf16_hi(w1));
                } else {
                    qb[ht][kk][0] = w0;
                    qb[ht][kk][1] = w1;
                }
            }
        }
    }

    const float sl = a.scale_log2 * ks;

    float acc[NH][C::KS][4];
#pragma unroll
    for (int ht = 0; ht < NH; ++ht)
#pragma unroll
        for (int md = 0; md < C::KS; ++md) acc[ht][md][0] = acc[ht][md][1] = acc[ht][md][2] = acc[ht][md][3] = 0.f;
    float mx[NH][2], ls[NH][2];  // running max (log2 units) and partial sum of heads 8 ht + 2t + e
#pragma unroll
    for (int ht = 0; ht < NH; ++ht) mx[ht][0] = mx[ht][1] = -INFINITY, ls[ht][0] = ls[ht][1] = 0.f;
    bool ok = true;
    int bad_pages = 0;
    int i = 0;
    int slot = 0;          // i % NSLOT
    uint32_t phase = 0u;   // (i / NSLOT) & 1

    // S^T = K Q^T for the 16 tokens of the page at kb: sc[ht] holds tokens
    // g (e = 0, 1) and g + 8 (e = 2, 3) of heads 8 ht + 2t + (e & 1).
    auto qk_page = [&](uint32_t kb, float (*sc)[4]) {
        if constexpr (KIND == kBf16) {
#pragma unroll
            for (int kk = 0; kk < C::KS; ++kk) {
                const int r = (lane & 7) + 8 * ((lane >> 3) & 1);
                const int col = 2 * (16 * kk + 8 * (lane >> 4));
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kb + swz<C::BOXB>(r, col), a0, a1, a2, a3);
#pragma unroll
                for (int ht = 0; ht < NH; ++ht) mma16816<false>(sc[ht], a0, a1, a2, a3, qb[ht][kk][0], qb[ht][kk][1]);
            }
        } else if constexpr (KIND == kFp8) {
            // rows g and g + 8: bytes [(D/4) t, (D/4)(t + 1)), one word per k-step
            uint32_t w[2][C::KS];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = g + 8 * hr;
                if constexpr (D == 128) {
                    const uint4 x0 = lds128(kb + swz<C::BOXB>(r, 32 * t));
                    const uint4 x1 = lds128(kb + swz<C::BOXB>(r, 32 * t + 16));
                    w[hr][0] = x0.x; w[hr][1] = x0.y; w[hr][2] = x0.z; w[hr][3] = x0.w;
                    w[hr][4] = x1.x; w[hr][5] = x1.y; w[hr][6] = x1.z; w[hr][7] = x1.w;
                } else {
                    const uint4 x0 = lds128(kb + swz<C::BOXB>(r, 16 * t));
                    w[hr][0] = x0.x; w[hr][1] = x0.y; w[hr][2] = x0.z; w[hr][3] = x0.w;
                }
            }
#pragma unroll
            for (int kk = 0; kk < C::KS; ++kk) {
                const uint32_t a0 = e4m3x2_to_f16x2(lo16(w[0][kk])), a1 = e4m3x2_to_f16x2(lo16(w[1][kk]));
                const uint32_t a2 = e4m3x2_to_f16x2(hi16(w[0][kk])), a3 = e4m3x2_to_f16x2(hi16(w[1][kk]));
#pragma unroll
                for (int ht = 0; ht < NH; ++ht) mma16816<true>(sc[ht], a0, a1, a2, a3, qb[ht][kk][0], qb[ht][kk][1]);
            }
        } else {
            // rows g and g + 8: bytes [(D/8) t, (D/8)(t + 1)), values
            // [(D/4) t, (D/4)(t + 1)) -- blocks 2t, 2t+1 (D = 128) or t
            constexpr int NW = D / 32;              // words of E2M1 pairs per row per thread
            const uint32_t kbs = kb + 2 * C::PAGE;  // K block scales [16][D/16]
            uint32_t w[2][NW], sA[2], sB[2];        // sA / sB: {s, s} of the first / second block
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = g + 8 * hr;
                if constexpr (D == 128) {
                    const uint4 x0 = lds128(kb + swz<C::BOXB>(r, 16 * t));
                    w[hr][0] = x0.x; w[hr][1] = x0.y; w[hr][2] = x0.z; w[hr][3] = x0.w;
                    const uint32_t s2 = e4m3x2_to_f16x2(static_cast<uint16_t>(lds16(kbs + r * C::SROW + 2 * t)));
                    sA[hr] = prmt(s2, s2, 0x1010u);
                    sB[hr] = prmt(s2, s2, 0x3232u);
                } else {
                    const uint2 x0 = lds64(kb + swz<C::BOXB>(r, 8 * t));
                    w[hr][0] = x0.x; w[hr][1] = x0.y;
                    const uint32_t s1 = lds8(kbs + r * C::SROW + t);
                    sA[hr] = sB[hr] = e4m3x2_to_f16x2(static_cast<uint16_t>(s1 | (s1 << 8)));
                }
            }
#pragma unroll
            for (int wi = 0; wi < NW; ++wi) {
                uint32_t ha[4], hb[4];
                e2m1x8_to_f16x2(w[0][wi], ha);
                e2m1x8_to_f16x2(w[1][wi], hb);
                const bool second = D == 128 && wi >= 2;  // words 2, 3 hold block 2t + 1
                const uint32_t fa = second ? sB[0] : sA[0];
                const uint32_t fb = second ? sB[1] : sA[1];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int kk = 2 * wi + j;
                    const uint32_t a0 = hmul2(ha[2 * j], fa), a2 = hmul2(ha[2 * j + 1], fa);
                    const uint32_t a1 = hmul2(hb[2 * j], fb), a3 = hmul2(hb[2 * j + 1], fb);
#pragma unroll
                    for (int ht = 0; ht < NH; ++ht)
                        mma16816<true>(sc[ht], a0, a1, a2, a3, qb[ht][kk][0], qb[ht][kk][1]);
                }
            }
        }
    };
    // O^T += V^T P^T for the page at vb; tokens at or past `valid` contribute
    // zero (their V bytes may be anything, so they are zeroed, not only
    // weighted 0). pb[ht] = P^T fragments of head tile ht.
    auto pv_page = [&](uint32_t vb, int valid, const uint32_t (*pb)[2], const uint32_t (*pl)[2]) {
        if constexpr (KIND == kBf16) {
            uint32_t mk0 = 0xFFFFFFFFu, mk1 = 0xFFFFFFFFu;
            if (valid < kPageSize) {
                mk0 = (2 * t < valid ? 0x0000FFFFu : 0u) | (2 * t + 1 < valid ? 0xFFFF0000u : 0u);
                mk1 = (2 * t + 8 < valid ? 0x0000FFFFu : 0u) | (2 * t + 9 < valid ? 0xFFFF0000u : 0u);
            }
#pragma unroll
            for (int md = 0; md < C::KS; ++md) {
                const int mi = lane >> 3;
                const int r = (lane & 7) + 8 * (mi >> 1);
                const int col = 2 * (16 * md + 8 * (mi & 1));
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(vb + swz<C::BOXB>(r, col), a0, a1, a2, a3);
                a0 &= mk0;
                a1 &= mk0;
                a2 &= mk1;
                a3 &= mk1;
#pragma unroll
                for (int ht = 0; ht < NH; ++ht) {
                    mma16816<false>(acc[ht][md], a0, a1, a2, a3, pb[ht][0], pb[ht][1]);
                    mma16816<false>(acc[ht][md], a0, a1, a2, a3, pl[ht][0], pl[ht][1]);
                }
            }
        } else if constexpr (KIND == kFp8) {
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
                // bytes {A d, B d, A d+1, B d+1}: tokens 2t / 2t+1 (p) and 2t+8 / 2t+9 (q)
                const uint32_t pl = prmt(va[0][wd], va[1][wd], 0x5140u);
                const uint32_t ph = prmt(va[0][wd], va[1][wd], 0x7362u);
                const uint32_t ql = prmt(va[2][wd], va[3][wd], 0x5140u);
                const uint32_t qh = prmt(va[2][wd], va[3][wd], 0x7362u);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t pw = j ? ph : pl, qw = j ? qh : ql;
                    const uint32_t a0 = e4m3x2_to_f16x2(lo16(pw)), a1 = e4m3x2_to_f16x2(hi16(pw));
                    const uint32_t a2 = e4m3x2_to_f16x2(lo16(qw)), a3 = e4m3x2_to_f16x2(hi16(qw));
#pragma unroll
                    for (int ht = 0; ht < NH; ++ht)
                        mma16816<true>(acc[ht][2 * wd + j], a0, a1, a2, a3, pb[ht][0], pb[ht][1]);
                }
            }
        } else {
            // thread g's share of each row: bytes [(D/16) g, (D/16)(g+1)),
            // values (D/8) g + [0, D/8) -- all in block g (D = 128) or g/2
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
                    const uint32_t a0 = hmul2(he[i2], s01), a1 = hmul2(ho[i2], s01);
                    const uint32_t a2 = hmul2(ge[i2], s89), a3 = hmul2(go[i2], s89);
#pragma unroll
                    for (int ht = 0; ht < NH; ++ht)
                        mma16816<true>(acc[ht][4 * wd + i2], a0, a1, a2, a3, pb[ht][0], pb[ht][1]);
                }
            }
        }
    };

    for (; i < nw; ++i) {
        if (i > 0 && (i & 31) == 0) {
            cur = nxt;
            nxt = load_batch((i >> 5) + 1);
        }
        const bool landed = mbar_wait_bounded(bar0 + 8 * slot, phase, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, landed)) {
            ok = false;
            break;
        }
        const int pid = page_id(i, i >> 5);
        const bool pid_ok = pid >= 0 && pid < num_pages;
        if (!pid_ok) ++bad_pages;
        const int p = p0 + warp + kWarps * i;
        const int valid = pid_ok ? min(kPageSize, L - p * kPageSize) : 0;
        if (valid > 0) {
            const uint32_t kslot = ring0 + slot * C::SLOT;
            float sc[NH][4];
#pragma unroll
            for (int ht = 0; ht < NH; ++ht) sc[ht][0] = sc[ht][1] = sc[ht][2] = sc[ht][3] = 0.f;
            qk_page(kslot, sc);

            // ---- online softmax (log2 domain) -------------------------------
            const bool v0 = g < valid, v1 = g + 8 < valid;
            float pr[NH][4], al[NH][2];
            bool moved = false;
#pragma unroll
            for (int ht = 0; ht < NH; ++ht) {
                float x[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) x[e] = ((e >> 1) ? v1 : v0) ? sc[ht][e] * sl : -INFINITY;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float pm = fmaxf(x[e], x[2 + e]);
                    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
                    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
                    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
                    const float nm = fmaxf(mx[ht][e], pm);
                    al[ht][e] = fast_exp2(mx[ht][e] - nm);
                    moved |= al[ht][e] != 1.f;
                    mx[ht][e] = nm;
                    pr[ht][e] = fast_exp2(x[e] - nm);
                    pr[ht][2 + e] = fast_exp2(x[2 + e] - nm);
                    ls[ht][e] = ls[ht][e] * al[ht][e] + (pr[ht][e] + pr[ht][2 + e]);
                }
            }
            // rescale the accumulators only when some head's max moved (after
            // the first pages it rarely does)
            if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
                for (int ht = 0; ht < NH; ++ht)
#pragma unroll
                    for (int md = 0; md < C::KS; ++md) {
                        acc[ht][md][0] *= al[ht][0];
                        acc[ht][md][1] *= al[ht][1];
                        acc[ht][md][2] *= al[ht][0];
                        acc[ht][md][3] *= al[ht][1];
                    }
            }
            // ---- P^T fragments: pack S^T's 8-token halves, transpose ----------
            // f16 weights keep 11 significant bits. bf16 keeps 8, too few
            // where the weighted values cancel (a relative error of 2^-9 of
            // each weight times |V|): bf16 weights are split into a rounded
            // term and the rounded rest, P = P_hi + P_lo to 2^-17, and V^T
            // meets both terms.
            uint32_t pb[NH][2], pl[NH][2];
#pragma unroll
            for (int ht = 0; ht < NH; ++ht) {
                uint32_t x0, x1;
                if constexpr (C::F16) {
                    x0 = pack_f16(pr[ht][0], pr[ht][1]);
                    x1 = pack_f16(pr[ht][2], pr[ht][3]);
                } else {
                    x0 = pack_bf16(pr[ht][0], pr[ht][1]);
                    x1 = pack_bf16(pr[ht][2], pr[ht][3]);
                    const uint32_t y0 = pack_bf16(pr[ht][0] - bf16_lo(x0), pr[ht][1] - bf16_hi(x0));
                    const uint32_t y1 = pack_bf16(pr[ht][2] - bf16_lo(x1), pr[ht][3] - bf16_hi(x1));
                    pl[ht][0] = movmatrix_trans(y0);
                    pl[ht][1] = movmatrix_trans(y1);
                }
                pb[ht][0] = movmatrix_trans(x0);
                pb[ht][1] = movmatrix_trans(x1);
            }
            pv_page(kslot + C::PAGE, valid, pb, pl);
        }

        // ---- refill the consumed slot with page i + NSLOT -------------------
        __syncwarp();
        const int nx = i + C::NSLOT;
        if (nx < nw) {
            const int pid2 = page_id(nx, i >> 5);
            fence_proxy_async_smem();  // this warp's reads of the slot before the copies' writes
            issue(slot, pid2);
        }
        if (++slot == C::NSLOT) {
            slot = 0;
            phase ^= 1u;
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
#pragma unroll
    for (int ht = 0; ht < NH; ++ht)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            ls[ht][e] += __shfl_xor_sync(0xffffffffu, ls[ht][e], 4);
            ls[ht][e] += __shfl_xor_sync(0xffffffffu, ls[ht][e], 8);
            ls[ht][e] += __shfl_xor_sync(0xffffffffu, ls[ht][e], 16);
        }
    __syncwarp();
    // [16][D + 8] partial sums (the 8-float pad spreads the rows over the
    // banks), then m[16], l[16]
    constexpr int CWS = D + 8;
    float* cw = reinterpret_cast<float*>(ring);
    float* cm = cw + 16 * CWS;
    float* cl = cm + 16;
    if (g == 0) {
#pragma unroll
        for (int ht = 0; ht < NH; ++ht)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                cm[8 * ht + 2 * t + e] = mx[ht][e];
                cl[8 * ht + 2 * t + e] = ls[ht][e];
            }
    }
#pragma unroll
    for (int ht = 0; ht < NH; ++ht)
#pragma unroll
        for (int md = 0; md < C::KS; ++md)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int h = 8 * ht + 2 * t + (e & 1);
                const int d = C::F16 ? (D / 8) * g + 2 * md + (e >> 1) : 16 * md + g + 8 * (e >> 1);
                cw[h * CWS + d] = acc[ht][md][e];
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

template <int D, int KIND, int NH>
cudaError_t launch_t(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int hnd, cudaStream_t s) {
    using C = Cfg<D, KIND>;
    auto kern = paged_decode_kernel<D, KIND, NH>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid = a.work ? dim3(static_cast<unsigned>(a.n_work * a.Hkv)) : dim3(a.num_splits, a.Hkv, a.B);
    return launch_dependent(kern, grid, dim3(kWarps * 32), C::SMEM, s, tk, tv, a, hnd);
}

template <int D, int KIND>
cudaError_t launch_g(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int hnd, cudaStream_t s) {
    return a.G > 8 ? launch_t<D, KIND, 2>(a, tk, tv, hnd, s) : launch_t<D, KIND, 1>(a, tk, tv, hnd, s);
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

int decode_ctas_per_sm(int D, int kind, int G) {
    (void)D;
    return ctas_per_sm(kind, G > 8 ? 2 : 1);
}

cudaError_t launch_paged_decode(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t s) {
    if (a.B == 0 || (a.work != nullptr && a.n_work == 0)) return cudaSuccess;
    const int hnd = a.layout == PKV_HND;
    if (a.D == 128) return launch_d<128>(a, tk, tv, hnd, s);
    if (a.D == 64) return launch_d<64>(a, tk, tv, hnd, s);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
