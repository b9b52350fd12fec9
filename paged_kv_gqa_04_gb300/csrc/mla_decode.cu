// mla_decode.cu -- paged multi-head latent attention (MLA) split-K decode
// for sm_103a, absorbed form.
//
// mainarch, MLA decode section: the cache holds one compressed latent per
// token (ckv, 512 values, FP8 E4M3) beside a 64-value positional part (kpe,
// BF16); the per-head projections are applied to the query before the cache
// is read, so every query head attends to the same cache rows: per-head dot
// scores over [ckv | kpe], a local softmax with exported LSE,
// softmax-weighted latent outputs (V = ckv), split-K over the sequence and a
// stage-2 merge of the partial records (pkv_lse_merge with D = 512).
//
// Work decomposition. One CTA per (split, sequence); four warps. The split's
// tokens stream through the CTA in chunks of 32 (half a 64-token page):
// warp 0's lanes issue TMA tile loads of a chunk -- four 32-row x 128-byte
// boxes of ckv and one 32-row x 128-byte box of kpe, 128-byte swizzle -- into
// a 4-slot ring of 20 KB slots, each tracked by an mbarrier. Warp w owns the
// latent columns [128w, 128w + 128) and the positional columns
// [16w, 16w + 16):
//   phase 1  partial scores S_w^T[32 tok x 8 h] over its columns
//            (mma.sync m16n8k16, the cache rows on M as in the GQA decode:
//            E4M3 -> f16 for ckv, bf16 ldmatrix for kpe), written to shared
//            memory;
//   barrier  (one per chunk; it also frees a consumed chunk's ring slot,
//            which warp 0 refills);
//   phase 2  every warp sums the four partials and runs the same online
//            softmax (so their running max and sum agree exactly);
//   phase 3  O_w^T[128 d x 8 h] += ckv^T[its 128 d x 32 tok] . P^T, the
//            E4M3 bytes paired by token with prmt.
// Each warp then writes its own 128 output columns: no cross-warp combine.
// The loop is software-pipelined: iteration c computes chunk c + 1's
// partial scores (phase 1) and chunk c's softmax and output (phases 2, 3)
// as two independent instruction streams, then meets the other warps at
// the chunk's one barrier (the partial-score exchange is double-buffered by
// chunk parity). Up to 16 heads per CTA (two head tiles of 8).
//
// Waits are bounded (about one second): a copy that never lands sets
// PKV_FLAG_WAIT_TIMEOUT, the CTA stops at the same chunk (the barrier
// agrees on it), waits (bounded) for its copies still in flight and exits.
#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kW = 4;                   // warps per CTA
constexpr int kCh = 32;                 // tokens per chunk
constexpr int kBox = kCh * 128;         // bytes of one 32-row x 128-byte box
constexpr int kSlot = 5 * kBox;         // four ckv boxes + one kpe box
constexpr uint64_t kWaitLimitNs = 1000000000ull;
#ifndef PKV_MLA_SLOTS_NH1
#define PKV_MLA_SLOTS_NH1 4
#endif
#ifndef PKV_MLA_CTAS_NH1
#define PKV_MLA_CTAS_NH1 2
#endif

// Up to 8 heads: PKV_MLA_CTAS_NH1 CTAs per SM with a PKV_MLA_SLOTS_NH1-slot
// ring; 16 heads (twice the registers): 2 CTAs, 4 slots.
template <int NH>
struct MlaCfg {
    static constexpr int NSLOT = NH == 1 ? PKV_MLA_SLOTS_NH1 : 4;  // ring slots
    static constexpr int CTAS = NH == 1 ? PKV_MLA_CTAS_NH1 : 2;
    static constexpr int PART = 2 * kW * 2 * NH * 32 * 16;  // partial scores: [parity][warp][mt, ht][lane] float4
    static constexpr int SMEM = NSLOT * kSlot + PART + NSLOT * 8 + 1024;
};

__device__ __forceinline__ uint32_t swz128(int r, int col) {
    return r * 128 + ((((col >> 4) & 7) ^ (r & 7)) << 4) + (col & 15);
}
__device__ __forceinline__ uint16_t lo16(uint32_t w) { return static_cast<uint16_t>(w & 0xFFFFu); }
__device__ __forceinline__ uint16_t hi16(uint32_t w) { return static_cast<uint16_t>(w >> 16); }

template <int NH>
__global__ void __launch_bounds__(kW * 32, MlaCfg<NH>::CTAS)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tckv, const __grid_constant__ CUtensorMap tkpe,
                      const MlaDecodeArgs a) {
    using C = MlaCfg<NH>;
    constexpr int kNSlot = C::NSLOT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem0 = smem_u32(smem);
    const uint32_t ring0 = smem0;
    const uint32_t part0 = smem0 + kNSlot * kSlot;
    const uint32_t bar0 = part0 + C::PART;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int s = blockIdx.x;
    const int b = blockIdx.y;
    const int H = a.H;

    // ---- this split's tokens ---------------------------------------------------
    int L = __ldg(a.seq_lens + b);
    const int cap = a.max_pages * kMlaPage;
    if (L < 0 || L > cap) {
        if (threadIdx.x == 0 && s == 0) flag_error(a.err, PKV_FLAG_SEQ_LEN_RANGE);
        L = L < 0 ? 0 : cap;
    }
    const int npages = (L + kMlaPage - 1) / kMlaPage;
    const int pps = (npages + a.num_splits - 1) / a.num_splits;
    const int p0 = s * pps;
    const int p1 = min(p0 + pps, npages);
    const int tok0 = p0 * kMlaPage;                                 // first logical token of the split
    const int ntok = p1 > p0 ? min(L, p1 * kMlaPage) - tok0 : 0;
    const int nch = (ntok + kCh - 1) / kCh;
    float* outp = a.out_partial + b * a.op_s0 + s * a.op_s1;
    float* lsep = a.lse_partial + b * a.lp_s0 + s * a.lp_s1;
    if (nch == 0) {  // empty split: (0, -inf)
        grid_dep_wait();
        grid_dep_launch();
        for (int i = threadIdx.x; i < H * kMlaDc; i += blockDim.x) outp[(i / kMlaDc) * a.op_s2 + (i % kMlaDc)] = 0.f;
        for (int i = threadIdx.x; i < H; i += blockDim.x) lsep[i] = -INFINITY;
        return;
    }
    const int32_t* bt = a.block_tables + b * a.bt_s0 + p0;
    auto page_of = [&](int c) -> int { return __ldg(bt + (c >> 1)); };  // chunk c lies in page p0 + c/2

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNSlot; ++i) mbar_init(bar0 + 8 * i, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tckv);
        tma_prefetch_desc(&tkpe);
    }
    __syncthreads();
    const uint64_t policy = l2_policy_evict_first();
    const int64_t num_pages = a.num_pages;

    // q and the cache may still be being written by the preceding grid.
    grid_dep_wait();
    grid_dep_launch();

    // Start the copies of chunk c into its slot; called by warp 0 (pid uniform).
    auto issue = [&](int c) {
        const int slot = c % kNSlot;
        const uint32_t bar = bar0 + 8 * slot;
        const int pid = page_of(c);
        if (pid < 0 || pid >= num_pages) {
            if (lane == 0) mbar_arrive(bar);  // completes the phase with no bytes; the chunk is skipped
            return;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar, kSlot);
        __syncwarp();
        const uint32_t dst = ring0 + slot * kSlot + lane * kBox;
        const int row0 = (c & 1) * kCh;
        if (lane < 4)
            tma_load_3d(dst, &tckv, bar, 128 * lane, row0, pid, policy);
        else if (lane == 4)
            tma_load_3d(dst, &tkpe, bar, 0, row0, pid, policy);
    };
    if (warp == 0)
        for (int c = 0; c < min(kNSlot, nch); ++c) issue(c);

    // ---- Q^T fragments (B operands) for this warp's columns --------------------
    // latent: k-step kk, k-rows 2t, 2t+1 (b0) / 2t+8, 2t+9 (b1) are columns
    // 128w + 32t + 4kk (+0, +1 / +2, +3) -- the order of the thread's ckv
    // bytes; positional: columns 16w + 2t (+8), natural order (ldmatrix).
    uint32_t qb[NH][8][2], qr[NH][2];
#pragma unroll
    for (int ht = 0; ht < NH; ++ht) {
        const int h = 8 * ht + g;
        const bool live = h < H;
        const uint16_t* ql = a.q_lat + b * a.ql_s0 + h * a.ql_s1 + 128 * warp + 32 * t;
        const uint16_t* qp = a.q_pe + b * a.qp_s0 + h * a.qp_s1 + 16 * warp + 2 * t;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t w0 = 0u, w1 = 0u;
            if (live) {
                w0 = __ldg(reinterpret_cast<const uint32_t*>(ql + 4 * kk));
                w1 = __ldg(reinterpret_cast<const uint32_t*>(ql + 4 * kk + 2));
            }
            qb[ht][kk][0] = pack_f16(bf16_lo(w0), bf16_hi(w0));
            qb[ht][kk][1] = pack_f16(bf16_lo(w1), bf16_hi(w1));
        }
        qr[ht][0] = live ? __ldg(reinterpret_cast<const uint32_t*>(qp)) : 0u;
        qr[ht][1] = live ? __ldg(reinterpret_cast<const uint32_t*>(qp + 8)) : 0u;
    }
    const float cks = __ldg(a.ckv_scale);
    const float sl = a.scale_log2;

    float acc[NH][8][4];
#pragma unroll
    for (int ht = 0; ht < NH; ++ht)
#pragma unroll
        for (int md = 0; md < 8; ++md) acc[ht][md][0] = acc[ht][md][1] = acc[ht][md][2] = acc[ht][md][3] = 0.f;
    float mx[NH][2], ls[NH][2];  // running max (log2 units), partial sums of heads 8 ht + 2t + e
#pragma unroll
    for (int ht = 0; ht < NH; ++ht) mx[ht][0] = mx[ht][1] = -INFINITY, ls[ht][0] = ls[ht][1] = 0.f;

    // chunk c: ring slot c % kNSlot, barrier phase (c / kNSlot) & 1, its
    // partial scores in parity buffer c & 1
    auto valid_of = [&](int c) -> int {  // tokens of chunk c (0: its page id is out of range)
        const int pid = page_of(c);
        return (pid >= 0 && pid < num_pages) ? min(kCh, ntok - c * kCh) : 0;
    };

    // ---- phase 1: partial scores of chunk c over this warp's columns -----------
    auto phase1 = [&](int c) {
        const uint32_t sb = ring0 + (c % kNSlot) * kSlot;
        const uint32_t ck = sb + warp * kBox;  // this warp's 128 ckv columns
        const uint32_t kp = sb + 4 * kBox;     // kpe box
        const uint32_t pw = part0 + (c & 1) * (kW * 2 * NH * 512);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            float sc[NH][4];
#pragma unroll
            for (int ht = 0; ht < NH; ++ht) sc[ht][0] = sc[ht][1] = sc[ht][2] = sc[ht][3] = 0.f;
            uint32_t w[2][8];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = 16 * mt + g + 8 * hr;
                const uint4 x0 = lds128(ck + swz128(r, 32 * t));
                const uint4 x1 = lds128(ck + swz128(r, 32 * t + 16));
                w[hr][0] = x0.x; w[hr][1] = x0.y; w[hr][2] = x0.z; w[hr][3] = x0.w;
                w[hr][4] = x1.x; w[hr][5] = x1.y; w[hr][6] = x1.z; w[hr][7] = x1.w;
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a0 = e4m3x2_to_f16x2(lo16(w[0][kk])), a1 = e4m3x2_to_f16x2(lo16(w[1][kk]));
                const uint32_t a2 = e4m3x2_to_f16x2(hi16(w[0][kk])), a3 = e4m3x2_to_f16x2(hi16(w[1][kk]));
#pragma unroll
                for (int ht = 0; ht < NH; ++ht) mma16816<true>(sc[ht], a0, a1, a2, a3, qb[ht][kk][0], qb[ht][kk][1]);
            }
#pragma unroll
            for (int ht = 0; ht < NH; ++ht)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[ht][e] *= cks;  // the ckv part carries the latent scale
            {
                const int r = 16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1);
                const int col = 2 * (16 * warp + 8 * (lane >> 4));
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kp + swz128(r, col), a0, a1, a2, a3);
#pragma unroll
                for (int ht = 0; ht < NH; ++ht) mma16816<false>(sc[ht], a0, a1, a2, a3, qr[ht][0], qr[ht][1]);
            }
#pragma unroll
            for (int ht = 0; ht < NH; ++ht)
                sts128(pw + ((warp * 2 * NH + mt * NH + ht) * 32 + lane) * 16, sc[ht][0], sc[ht][1], sc[ht][2],
                       sc[ht][3]);
        }
    };

    // ---- phases 2 and 3 of chunk c: total scores and online softmax (every
    // warp the same), then O^T += ckv^T P^T over this warp's 128 columns ------
    auto phase23 = [&](int c, int valid) {
        const uint32_t ck = ring0 + (c % kNSlot) * kSlot + warp * kBox;
        const uint32_t pw = part0 + (c & 1) * (kW * 2 * NH * 512);
        float pr[2][NH][4];
        float al[NH][2];
        bool moved = false;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int ht = 0; ht < NH; ++ht) {
                float4 tot = lds128f(pw + ((0 * 2 * NH + mt * NH + ht) * 32 + lane) * 16);
#pragma unroll
                for (int w = 1; w < kW; ++w) {
                    const float4 y = lds128f(pw + ((w * 2 * NH + mt * NH + ht) * 32 + lane) * 16);
                    tot.x += y.x; tot.y += y.y; tot.z += y.z; tot.w += y.w;
                }
                const bool v0 = 16 * mt + g < valid, v1 = 16 * mt + g + 8 < valid;
                pr[mt][ht][0] = v0 ? tot.x * sl : -INFINITY;
                pr[mt][ht][1] = v0 ? tot.y * sl : -INFINITY;
                pr[mt][ht][2] = v1 ? tot.z * sl : -INFINITY;
                pr[mt][ht][3] = v1 ? tot.w * sl : -INFINITY;
            }
#pragma unroll
        for (int ht = 0; ht < NH; ++ht)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float pm = fmaxf(fmaxf(pr[0][ht][e], pr[0][ht][2 + e]), fmaxf(pr[1][ht][e], pr[1][ht][2 + e]));
                pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
                pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
                pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
                const float nm = fmaxf(mx[ht][e], pm);
                al[ht][e] = fast_exp2(mx[ht][e] - nm);
                moved |= al[ht][e] != 1.f;
                mx[ht][e] = nm;
                float sum = 0.f;
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    pr[mt][ht][e] = fast_exp2(pr[mt][ht][e] - nm);
                    pr[mt][ht][2 + e] = fast_exp2(pr[mt][ht][2 + e] - nm);
                    sum += pr[mt][ht][e] + pr[mt][ht][2 + e];
                }
                ls[ht][e] = ls[ht][e] * al[ht][e] + sum;
            }
        if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
            for (int ht = 0; ht < NH; ++ht)
#pragma unroll
                for (int md = 0; md < 8; ++md) {
                    acc[ht][md][0] *= al[ht][0];
                    acc[ht][md][1] *= al[ht][1];
                    acc[ht][md][2] *= al[ht][0];
                    acc[ht][md][3] *= al[ht][1];
                }
        }
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            uint32_t pb[NH][2];
#pragma unroll
            for (int ht = 0; ht < NH; ++ht) {
                pb[ht][0] = movmatrix_trans(pack_f16(pr[kb][ht][0], pr[kb][ht][1]));
                pb[ht][1] = movmatrix_trans(pack_f16(pr[kb][ht][2], pr[kb][ht][3]));
            }
            // thread g: columns 128w + 16g .. +15 of tokens 16kb + 2t, 2t+1, 2t+8, 2t+9
            uint32_t va[4][4];
            const int rows[4] = {16 * kb + 2 * t, 16 * kb + 2 * t + 1, 16 * kb + 2 * t + 8, 16 * kb + 2 * t + 9};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 xv = lds128(ck + swz128(rows[q], 16 * g));
                const bool in = rows[q] < valid;  // bytes past the sequence end may be anything
                va[q][0] = in ? xv.x : 0u;
                va[q][1] = in ? xv.y : 0u;
                va[q][2] = in ? xv.z : 0u;
                va[q][3] = in ? xv.w : 0u;
            }
#pragma unroll
            for (int wd = 0; wd < 4; ++wd) {
                const uint32_t pl = prmt(va[0][wd], va[1][wd], 0x5140u);
                const uint32_t ph = prmt(va[0][wd], va[1][wd], 0x7362u);
                const uint32_t ql = prmt(va[2][wd], va[3][wd], 0x5140u);
                const uint32_t qh = prmt(va[2][wd], va[3][wd], 0x7362u);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t pwd = j ? ph : pl, qwd = j ? qh : ql;
                    const uint32_t a0 = e4m3x2_to_f16x2(lo16(pwd)), a1 = e4m3x2_to_f16x2(hi16(pwd));
                    const uint32_t a2 = e4m3x2_to_f16x2(lo16(qwd)), a3 = e4m3x2_to_f16x2(hi16(qwd));
#pragma unroll
                    for (int ht = 0; ht < NH; ++ht)
                        mma16816<true>(acc[ht][2 * wd + j], a0, a1, a2, a3, pb[ht][0], pb[ht][1]);
                }
            }
        }
    };

    // ---- software pipeline: chunk c + 1's partial scores are computed while
    // chunk c's softmax and output accumulate; one barrier per chunk --------
    int bad = 0;
    int v_cur = valid_of(0);
    bool landed = mbar_wait_bounded(bar0, 0u, kWaitLimitNs);
    if (v_cur > 0) phase1(0);
    if (v_cur == 0 && threadIdx.x == 0) ++bad;
    bool ok = __syncthreads_and(landed) != 0;
    int first_pending = 0;  // the oldest chunk whose copies may still be in flight
    int c = 0;
    if (ok) {
        for (; c < nch; ++c) {
            const int cn = c + 1;
            landed = true;
            int v_next = 0;
            if (cn < nch) {
                landed = mbar_wait_bounded(bar0 + 8 * (cn % kNSlot), (cn / kNSlot) & 1, kWaitLimitNs);
                v_next = valid_of(cn);
                if (v_next > 0) phase1(cn);
            }
            if (v_cur > 0) phase23(c, v_cur);
            // the partials of chunk c + 1 are complete, every warp is done
            // with chunk c (its slot may be refilled), and all agree on
            // whether chunk c + 1's copies landed
            ok = __syncthreads_and(landed) != 0;
            if (!ok) {
                first_pending = cn;
                break;
            }
            if (cn < nch && v_next == 0 && threadIdx.x == 0) ++bad;
            if (warp == 0 && c + kNSlot < nch) {
                fence_proxy_async_smem();  // the CTA's reads of the slot before the copies' writes
                issue(c + kNSlot);
            }
            v_cur = v_next;
        }
    }

    if (!ok) {
        // A copy never landed: record it, then wait (bounded) for the copies
        // still in flight before exiting.
        if (threadIdx.x == 0) flag_error(a.err, PKV_FLAG_WAIT_TIMEOUT);
        if (warp == 0) {
            const int last = min(c + kNSlot, nch);
            for (int j = first_pending; j < last; ++j)
                (void)mbar_wait_bounded(bar0 + 8 * (j % kNSlot), (j / kNSlot) & 1, kWaitLimitNs);
        }
        __syncthreads();
    }
    if (bad) flag_error(a.err, PKV_FLAG_PAGE_RANGE);

    // ---- epilogue: this warp's 128 columns of every head ------------------------
#pragma unroll
    for (int ht = 0; ht < NH; ++ht)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            ls[ht][e] += __shfl_xor_sync(0xffffffffu, ls[ht][e], 4);
            ls[ht][e] += __shfl_xor_sync(0xffffffffu, ls[ht][e], 8);
            ls[ht][e] += __shfl_xor_sync(0xffffffffu, ls[ht][e], 16);
        }
#pragma unroll
    for (int ht = 0; ht < NH; ++ht)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = 8 * ht + 2 * t + e;
            if (h >= H) continue;
            const bool empty = !(ls[ht][e] > 0.f);
            const float inv = empty ? 0.f : cks / ls[ht][e];
            float* orow = outp + h * a.op_s2 + 128 * warp + 16 * g;
#pragma unroll
            for (int md = 0; md < 8; ++md)
                *reinterpret_cast<float2*>(orow + 2 * md) = make_float2(acc[ht][md][e] * inv, acc[ht][md][2 + e] * inv);
            if (warp == 0 && g == 0)
                lsep[h] = empty ? -INFINITY : (mx[ht][e] + __log2f(ls[ht][e])) * 0.69314718055994530942f;
        }
}

template <int NH>
cudaError_t launch_t(const MlaDecodeArgs& a, const CUtensorMap& tckv, const CUtensorMap& tkpe, cudaStream_t s) {
    auto kern = mla_decode_kernel<NH>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, MlaCfg<NH>::SMEM);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3(a.num_splits, a.B), dim3(kW * 32), MlaCfg<NH>::SMEM, s, tckv, tkpe, a);
}

}  // namespace

int mla_decode_ctas_per_sm(int H) { return H > 8 ? MlaCfg<2>::CTAS : MlaCfg<1>::CTAS; }

cudaError_t launch_mla_decode(const MlaDecodeArgs& a, const CUtensorMap& tckv, const CUtensorMap& tkpe,
                              cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    return a.H > 8 ? launch_t<2>(a, tckv, tkpe, s) : launch_t<1>(a, tckv, tkpe, s);
}

}  // namespace pkv
