// mla_decode.cu -- paged multi-head latent attention (MLA) split-K decode
// for sm_103a on the fifth-generation tensor cores (tcgen05), absorbed form.
//
// mainarch, MLA decode section: the cache holds one compressed latent per
// token (ckv, 512 values, FP8 E4M3) beside a 64-value positional part (kpe,
// BF16); the per-head projections are applied to the query before the cache
// is read, so every query head attends to the same cache rows: per-head dot
// scores over [ckv | kpe], a local softmax with exported LSE,
// softmax-weighted latent outputs (V = ckv), split-K over the sequence and a
// stage-2 merge of the partial records (pkv_lse_merge with D = 512).
//
// The tensor cores read the E4M3 cache bytes as the TMA copies land them:
// nothing is converted on the CUDA cores.
//
// Work decomposition. Persistent CTAs, two per SM (106 KB of shared memory,
// 256 tensor-memory columns each), six warps in three roles. The work items
// are the (sequence, split) pairs, dealt to the CTAs in rounds of `grid`
// schedule positions: for batches up to 64 the positions walk the sequences
// longest first and every other round runs in reverse (so a CTA that drew
// one of the longest splits draws one of the shortest next); larger batches
// go round-robin (CTA k takes items k, k + grid, ...). A split's tokens go
// through the CTA two pages (128 tokens, the MMA M) at a time ("chunk"), one
// chunk in shared memory at a time; the copies run on across items, so only
// a CTA's first chunk waits for a cold start, and the two CTAs of an SM
// overlap each other's waits.
//
//   warp 0, copies    TMA tile loads with 128-byte swizzle into the chunk
//                     buffer: per page four 64-row x 128-byte boxes of ckv
//                     (one per 128-value column block) and one of kpe; the
//                     buffer holds ckv as [4 blocks][128 rows][128 B] and
//                     kpe as [128 rows][128 B] (80 KB). The next chunk is
//                     prefetched into L2 (cp.async.bulk.prefetch): the
//                     first chunk before the wait on the preceding grid (a
//                     prefetch reads through L2, which the preceding grid's
//                     writes also go through), the read-ahead only once the
//                     first chunk has landed.
//   warp 1, MMA       the whole warp runs the issue loop; one elected lane
//                     issues (elect.sync):
//                       S^T[128 tok x 32]   = ckv . Q8^T    (kind::f8f6f4, E4M3 x E4M3, K = 512)
//                       Spe^T[128 tok x 16] = kpe . q_pe^T  (kind::f16, bf16, K = 64)
//                     then, once P is ready,
//                       O^T[512 d x 48]    += ckv^T . P8^T  (E4M3 x E5M2, K = 128)
//                     as four M = 128 MMAs per 32-token step: the buffer's
//                     ckv bytes, read as an MN-major operand, are V^T.
//                     O accumulates in tensor memory over the whole split.
//   warps 2-5, softmax  (lane = token: warp w holds tokens 32(w%4) + 0..31)
//                     scores from tensor memory, per-head chunk maxima
//                     (redux.sync, a 4-warp exchange), P, its E5M2 terms to
//                     shared memory, the running sums; per item the next
//                     item's queries (so its scores overlap) and then the
//                     epilogue; the (0, -inf) records of empty splits.
//                     Query staging: warp q takes heads 4q .. 4q + 3 and
//                     reads whole 512-byte stretches of each row. Epilogue:
//                     l over the warp's tokens by recursive halving, one
//                     thread per head forms ckv_scale / (2^7 l) and the LSE,
//                     O is read from tensor memory two blocks per wait.
//
// The kernel has two instantiations by the heads its softmax warps handle:
// NH = 8 when H <= 8 (scores, weights, rescale and epilogue on 8 of each
// 16-column group; the P8 rows of heads 8-15 are zeroed once), else 16. The
// MMA shapes keep 16 head slots either way.
//
// Per chunk the steps are serial: copy -> S -> P -> P . V -> the buffer is
// free for the next copy. So the next chunk's scores never overwrite S
// before it was read, P is never rewritten before P . V read it, O is never
// scaled while P . V runs, and an item's first P . V (which starts O anew)
// comes after the softmax warps read the previous item's O.
//
// The operands, in FP8:
//   Q8: q_lat = 2^-k_h (t1 + t2) per head h, t1 = E4M3(2^k_h q),
//       t2 = E4M3(2^k_h q - t1), 2^k_h the largest power of two with
//       2^k_h max|q_h| <= 448. A bf16 value has 8 significant bits and t1
//       keeps 4, so t2 holds the rest exactly wherever its last bit is not
//       below E4M3's smallest step 2^-9: for 2^k_h |q| >= 2^-2, i.e. every
//       value within 2^9 of the head's largest; below, the error is at most
//       2^-10 2^-k_h. Rows 0-15 of Q8 are the t1 of heads 0-15, rows 16-31
//       the t2; S = 2^-k_h (S[:, h] + S[:, 16 + h]).
//   P8: the weight P = 2^(s - m) (<= 2^8, see below) as x = 2^7 P rounded
//       to f16, split into three E5M2 terms each rounded to nearest:
//       e1 = E5M2(x), e2 = E5M2(x - e1), e3 = E5M2(x - e1 - e2) (E5M2 is the
//       high byte of an f16: the remainders are f16, exact). For x >= 2^-6
//       the three sum to x exactly (the weight's error is the f16 rounding,
//       2^-11 relative); below, within 2^-17. Rows 16t + h of P8 hold term t
//       of head h; O is the sum of the three 16-column groups, times 2^-7.
//
// The online softmax keeps a reference maximum m per head that moves only
// when a chunk's maximum exceeds it by more than 8 (so P <= 2^8 and 2^7 P
// stays below E5M2's 57344); when it moves, the softmax warps scale O in
// tensor memory (tcgen05.ld / st) and the running sums by 2^(m_old - m_new)
// before handing P over. Tokens that take no part (past the sequence end,
// or on a page whose id is out of range) get P = 0, and their ckv rows are
// zeroed in shared memory before P . V reads them (a 0 weight times a NaN
// byte would poison the sum).
//
// Every hand-off is an mbarrier (the TMA copies' byte counts,
// tcgen05.commit, warp arrivals). Tensor memory: S (48 columns) and O
// (4 x 48 columns). Up to 16 heads; missing heads get zero queries and are
// not written.
//
// Waits are bounded (about one second). A role that gives up sets
// PKV_FLAG_WAIT_TIMEOUT and a CTA-wide abort flag that ends the other
// roles' waits; the four softmax warps agree on stopping through their
// barrier's AND; the copy and MMA roles wait (bounded) for their own
// operations in flight; the CTA then frees its tensor memory and exits.
#include <algorithm>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kT = 2 * kMlaPage;  // tokens per chunk (two pages), the MMA M
constexpr int kN = 16;            // heads per CTA
constexpr int kThreads = 192;
constexpr int kCtasPerSm = 2;
constexpr int kPrefetch = 1;      // chunks read into L2 ahead of the copy (measured best of 0-3)
constexpr int kWarpCopy = 0, kWarpMma = 1, kWarpSm = 2;
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// shared memory, byte offsets from a 1024-byte-aligned base
constexpr int kCkvBlock = kT * 128;               // one 128-value column block of a chunk
constexpr int kPageRows = kMlaPage * 128;         // a page's rows in one block
constexpr int kSlotCkv = 4 * kCkvBlock;
constexpr int kSlotBytes = kSlotCkv + kT * 128;   // + kpe [128 rows][128 B]
constexpr int kOffSlot = 0;
constexpr int kOffQ = kOffSlot + kSlotBytes;         // Q8 E4M3 [4 blocks][32 rows][128 B]
constexpr int kQBlock = 32 * 128;
constexpr int kOffQp = kOffQ + 4 * kQBlock;           // q_pe bf16 [16 rows][128 B]
constexpr int kOffP = kOffQp + kN * 128;              // P8 E5M2 [48 rows][128 B]
constexpr int kPBytes = 48 * 128;
constexpr int kRedBytes = 4 * kN * 4;                 // [4 warps][16 heads] floats
constexpr int kOffMax = kOffP + kPBytes;              // per-warp chunk maxima
constexpr int kOffSum = kOffMax + kRedBytes;          // per-warp sums
constexpr int kOffQs = kOffSum + kRedBytes;           // [16] floats: ckv_scale 2^-k_h
constexpr int kSortMaxB = 64;                         // batches ordered by length up to this size
constexpr int kOffOrder = kOffQs + kN * 4;            // [64] int16: sequences, longest first
constexpr int kOffBar = kOffOrder + kSortMaxB * 2;
enum : int { bFull = 0, bFree, bSFull, bPFull, bOFull, bQFull, kNumBars };
constexpr int kOffMisc = kOffBar + 8 * kNumBars;      // tensor-memory base, abort flag
constexpr int kSmem = kOffMisc + 16 + 1024;           // + alignment slack
static_assert(kCtasPerSm * (kSmem + 1024) <= 233472, "shared memory per SM");
static_assert(kSlotBytes % 1024 == 0 && kOffQ % 1024 == 0 && kOffQp % 1024 == 0 && kOffP % 1024 == 0 &&
                  kPBytes % 1024 == 0,
              "128-byte-swizzled tiles start on 1024-byte boundaries");

// tensor-memory columns
constexpr uint32_t kTmemCols = 256;  // per CTA: two CTAs fill an SM's 512
constexpr uint32_t kColS = 0;        // [S t1 | S t2 | Spe] (48)
constexpr uint32_t kColO = 64;       // 4 blocks of 128 latent rows x [3 terms x 16 heads]
constexpr float kRescaleLog2 = 8.f;  // P = 2^(s - m) <= 2^8
constexpr float kPScale = 128.f;     // P8 holds 2^7 P

constexpr uint32_t kIdescQk = umma_idesc(kT, 32, 0, 0, false, false);  // E4M3 x E4M3
constexpr uint32_t kIdescPe = umma_idesc(kT, kN, 1, 1, false, false);  // bf16 x bf16
constexpr uint32_t kIdescPv = umma_idesc(kT, 48, 0, 1, true, false);   // E4M3 (MN-major) x E5M2

__device__ __forceinline__ uint64_t desc_k(uint32_t addr) { return umma_desc_sw128(addr, 16, 1024); }

// Wait for a phase; false after about a second or once another role has
// given up.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const volatile int* abort_flag) {
    return mbar_wait_or_abort(bar, parity, abort_flag, kWaitLimitNs);
}

// One work item: split s of sequence b (items are numbered b * S + s, or
// are the entries of a split plan's work list).
struct Item {
    int b, s;
    int npg;              // pages of the split
    int ntok;             // tokens of the split
    int nch;              // chunks of the split
    bool bad_len;         // seq_lens[b] outside [0, block-table width x page]
    bool planless;        // a plan entry outside the batch or the records: no record, no work
    bool plan_bad;        // S_b outside [1, records] (clamped) or s >= S_b (an empty record)
    const int32_t* bt;    // the split's block-table entries
};

__device__ __forceinline__ Item item_of(const MlaDecodeArgs& a, int it) {
    Item x;
    int S = a.num_splits;
    x.planless = x.plan_bad = false;
    if (a.work == nullptr) {
        x.b = it / a.num_splits;
        x.s = it - x.b * a.num_splits;
    } else {
        const int e = __ldg(a.work + 2 * it);
        x.b = e >> 12;
        x.s = e & 0xFFF;
        if (x.b < 0 || x.b >= a.B || x.s >= a.num_splits) {
            x.planless = true;
            x.b = 0;
            x.npg = x.ntok = x.nch = 0;
            x.bad_len = false;
            x.bt = a.block_tables;
            return x;
        }
        const int r = __ldg(a.splits_per_seq + x.b);
        S = min(max(r, 1), a.num_splits);
        x.plan_bad = r != S || x.s >= S;
    }
    const int L0 = __ldg(a.seq_lens + x.b);
    const int cap = a.max_pages * kMlaPage;
    x.bad_len = L0 < 0 || L0 > cap;
    const int L = min(max(L0, 0), cap);
    const int npages = (L + kMlaPage - 1) / kMlaPage;
    const int pps = (npages + S - 1) / S;
    const int p0 = x.s * pps;
    const int p1 = min(p0 + pps, npages);
    x.npg = max(p1 - p0, 0);
    x.ntok = p1 > p0 ? min(L, p1 * kMlaPage) - p0 * kMlaPage : 0;
    x.nch = (x.ntok + kT - 1) / kT;
    x.bt = a.block_tables + x.b * a.bt_s0 + p0;
    return x;
}

// page id of page pg of the item if it exists and is in range, else -1
__device__ __forceinline__ int page_of(const Item& x, int pg, int64_t num_pages) {
    if (pg >= x.npg) return -1;
    const int pid = __ldg(x.bt + pg);
    return (pid >= 0 && pid < num_pages) ? pid : -1;
}

// The CTA's j-th item (n_items past the end). Schedule positions are dealt
// to the CTAs in rounds of gridDim.x. Without an order (batches above
// kSortMaxB) position p is item p, so CTA k takes k, k + G, k + 2G, ...
// With one, the positions walk the sequences longest first (each one's
// splits in turn) and every other round is dealt in reverse, so a CTA that
// drew one of the longest splits draws one of the shortest next.
__device__ __forceinline__ int slot_item(const MlaDecodeArgs& a, const int16_t* order, int j, int n_items) {
    const int G = gridDim.x, k = blockIdx.x;
    if (a.work != nullptr) order = nullptr;  // a plan's items come in its own order
    const int64_t p = static_cast<int64_t>(j) * G + ((order != nullptr && (j & 1)) ? G - 1 - k : k);
    if (p >= n_items) return n_items;  // only the last round is partial: nothing follows
    if (order == nullptr) return static_cast<int>(p);
    const int r = static_cast<int>(p) / a.num_splits;
    return order[r] * a.num_splits + (static_cast<int>(p) - r * a.num_splits);
}

// Position in this CTA's sequence of chunks: chunk c of its j-th item `it`
// (it >= n_items: past the end). Items without tokens are skipped.
struct Cursor {
    int j;
    int it;
    int c;
    Item x;
};
__device__ __forceinline__ void settle(const MlaDecodeArgs& a, const int16_t* order, Cursor& u, int n_items) {
    u.c = 0;
    for (;; ++u.j) {
        u.it = slot_item(a, order, u.j, n_items);
        if (u.it >= n_items) return;
        u.x = item_of(a, u.it);
        if (u.x.nch > 0) return;
    }
}
__device__ __forceinline__ void step(const MlaDecodeArgs& a, const int16_t* order, Cursor& u, int n_items) {
    if (++u.c >= u.x.nch) {
        ++u.j;
        settle(a, order, u, n_items);
    }
}

// NH columns (one per head) of a warp's tensor-memory lanes: the heads the
// softmax warps handle, 8 when H <= 8, else 16.
template <int NH>
__device__ __forceinline__ void tmem_ld_heads(uint32_t t, uint32_t (&r)[NH]) {
    if constexpr (NH == 16)
        tmem_ld16(t, r);
    else
        tmem_ld8(t, r);
}
template <int NH>
__device__ __forceinline__ void tmem_st_heads(uint32_t t, const uint32_t (&r)[NH]) {
    if constexpr (NH == 16)
        tmem_st16(t, r);
    else
        tmem_st8(t, r);
}

template <int NH>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tckv, const __grid_constant__ CUtensorMap tkpe,
                      const MlaDecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s0 = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return s0 + kOffBar + 8 * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int H = a.H;
    const int n_items = a.work != nullptr ? static_cast<int>(a.n_work) : a.B * a.num_splits;
    const int64_t num_pages = a.num_pages;

    if (threadIdx.x == 0) {
        mbar_init(bar(bFull), 1);
        mbar_init(bar(bFree), 1);
        mbar_init(bar(bSFull), 1);
        mbar_init(bar(bPFull), 4);
        mbar_init(bar(bOFull), 1);
        mbar_init(bar(bQFull), 4);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tckv);
        tma_prefetch_desc(&tkpe);
    }
    // At most two CTAs per SM (shared memory), each holding half of the
    // tensor memory, so the allocation never waits for another CTA.
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    // The schedule order: sequences by page count, longest first, ties by
    // index (index inputs only, read before the grid-dependency wait like
    // the L2 read-ahead below).
    int16_t* order_tab = reinterpret_cast<int16_t*>(smem + kOffOrder);
    if (warp == kWarpCopy && a.B <= kSortMaxB && a.work == nullptr) {
        const int cap = a.max_pages * kMlaPage;
        int key[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int b = lane + 32 * t;
            key[t] = b < a.B ? (min(max(__ldg(a.seq_lens + b), 0), cap) + kMlaPage - 1) / kMlaPage : -1;
        }
        int rank[2] = {0, 0};
        for (int b2 = 0; b2 < a.B; ++b2) {
            const int kb = __shfl_sync(0xffffffffu, b2 < 32 ? key[0] : key[1], b2 & 31);
#pragma unroll
            for (int t = 0; t < 2; ++t)
                rank[t] += (kb > key[t] || (kb == key[t] && b2 < lane + 32 * t)) ? 1 : 0;
        }
#pragma unroll
        for (int t = 0; t < 2; ++t)
            if (lane + 32 * t < a.B) order_tab[rank[t]] = static_cast<int16_t>(lane + 32 * t);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int16_t* order = (a.B <= kSortMaxB && a.work == nullptr) ? order_tab : nullptr;

    // L2 read-ahead of one chunk (lanes 0-4: its first page, 8-12: second)
    auto prefetch_at = [&](const Cursor& u) {
        const int half = lane >> 3, j = lane & 7;
        if (u.it < n_items && half < 2 && j < 5) {
            const int id = page_of(u.x, 2 * u.c + half, num_pages);
            if (id >= 0) {
                if (j < 4)
                    tma_prefetch_3d(&tckv, 128 * j, 0, id);
                else
                    tma_prefetch_3d(&tkpe, 0, 0, id);
            }
        }
    };
    // L2 read-ahead of the queries of item it (lane h < 16: q_lat row h,
    // 16 + h: q_pe row h), for 16-byte aligned rows
    auto prefetch_q = [&](int it) {
        if (it >= n_items) return;
        const int bq = a.work != nullptr ? min(max(__ldg(a.work + 2 * it) >> 12, 0), a.B - 1) : it / a.num_splits;
        const int h = lane & 15;
        if (h < H) {
            const void* r = lane < 16 ? static_cast<const void*>(a.q_lat + bq * a.ql_s0 + h * a.ql_s1)
                                      : static_cast<const void*>(a.q_pe + bq * a.qp_s0 + h * a.qp_s1);
            if ((reinterpret_cast<uintptr_t>(r) & 15) == 0) bulk_prefetch_l2(r, lane < 16 ? 2 * kMlaDc : 2 * kMlaDr);
        }
    };
    // The first chunk and queries go into L2 while the preceding grid may
    // still run (a prefetch loads nothing into this CTA; the index inputs
    // are this call's own).
    Cursor cur;
    cur.j = 0;
    if (warp == kWarpCopy) {
        settle(a, order, cur, n_items);
        prefetch_at(cur);
        prefetch_q(cur.it);
    }

    // q and the cache may still be being written by the preceding grid.
    grid_dep_wait();
    grid_dep_launch();

    auto give_up = [&]() {
        *abort_flag = 1;
        flag_error(a.err, PKV_FLAG_WAIT_TIMEOUT);
    };
    // warp-uniform bounded wait; a failure stops the other roles too
    auto warp_wait = [&](uint32_t bb, uint32_t par) -> bool {
        const bool r = __all_sync(0xffffffffu, wait_or_abort(bb, par, abort_flag));
        if (!r && lane == 0) give_up();
        return r;
    };

    if (warp == kWarpCopy) {
        // ======================= copies ===========================================
        const uint64_t policy = l2_policy_evict_first();
        Cursor pf = cur;  // the L2 read-ahead, kPrefetch chunks ahead of the copy
        int g = 0, issued = 0;  // chunks of this CTA whose copies were started
        for (; cur.it < n_items; step(a, order, cur, n_items), ++g) {
            if (g >= 1 && !warp_wait(bar(bFree), (g - 1) & 1)) break;  // chunk g - 1's P . V is done
            const int pa = 2 * cur.c, pb = pa + 1;
            const int ida = page_of(cur.x, pa, num_pages), idb = page_of(cur.x, pb, num_pages);
            if (lane == 0 && (ida < 0 || (pb < cur.x.npg && idb < 0))) flag_error(a.err, PKV_FLAG_PAGE_RANGE);
            const uint32_t fb = bar(bFull);
            const uint32_t bytes = (ida >= 0 ? 5 * kPageRows : 0) + (idb >= 0 ? 5 * kPageRows : 0);
            if (lane == 0) {
                if (bytes)
                    mbar_arrive_expect_tx(fb, bytes);
                else
                    mbar_arrive(fb);  // nothing to load: the phase completes at once
            }
            __syncwarp();
            const uint32_t sb = s0 + kOffSlot;
            const int half = lane >> 3, j = lane & 7;  // lanes 0-4: first page, 8-12: second
            const int id = half ? idb : ida;
            if (half < 2 && id >= 0 && j < 5) {
                if (j < 4)
                    tma_load_3d(sb + j * kCkvBlock + half * kPageRows, &tckv, fb, 128 * j, 0, id, policy);
                else
                    tma_load_3d(sb + kSlotCkv + half * kPageRows, &tkpe, fb, 0, 0, id, policy);
            }
            __syncwarp();
            issued = g + 1;
            if (cur.c == 0) prefetch_q(slot_item(a, order, cur.j + 1, n_items));  // the next item's queries
            if (g == 0) {
                // Every CTA's first chunk is requested before any read-ahead,
                // so none waits behind the other CTAs' later chunks.
                step(a, order, pf, n_items);
                if (pf.it < n_items && !warp_wait(fb, 0)) break;
                for (int k = 1; k <= kPrefetch; ++k) {
                    prefetch_at(pf);
                    if (k < kPrefetch) step(a, order, pf, n_items);
                }
            } else {
                step(a, order, pf, n_items);
                prefetch_at(pf);
            }
        }
        // The copies started land before the CTA may exit: wait (bounded)
        // for the newest phase (at once on the normal path).
        if (lane == 0 && issued > 0) (void)mbar_wait_bounded(bar(bFull), (issued - 1) & 1, kWaitLimitNs);
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ======================= tensor-core issue ================================
        int n_qk = 0, n_pv = 0;  // chunks whose MMAs were issued
        auto qk = [&](int g) -> bool {
            if (!warp_wait(bar(bFull), g & 1)) return false;
            tc_fence_after();
            const uint32_t sb = s0 + kOffSlot;
            const uint32_t dS = tmem + kColS;
#pragma unroll
            for (int k = 0; k < kMlaDc / 32; ++k)
                umma_f8_warp(dS, desc_k(sb + (k >> 2) * kCkvBlock + (k & 3) * 32),
                             desc_k(s0 + kOffQ + (k >> 2) * kQBlock + (k & 3) * 32), kIdescQk, k > 0);
#pragma unroll
            for (int k = 0; k < kMlaDr / 16; ++k)
                umma_f16_warp(dS + 32, desc_k(sb + kSlotCkv + k * 32), desc_k(s0 + kOffQp + k * 32), kIdescPe, k > 0);
            umma_commit_warp(bar(bSFull));
            n_qk = g + 1;
            return true;
        };
        // P . V of chunk g, the item's chunk c (c = 0 starts the item's O;
        // the item before has read its O by then: its epilogue precedes the
        // softmax warps' P of this chunk)
        auto pv = [&](int g, int c) -> bool {
            if (!warp_wait(bar(bPFull), g & 1)) return false;
            tc_fence_after();
            const uint32_t sb = s0 + kOffSlot;
            const uint32_t pb = s0 + kOffP;
#pragma unroll
            for (int k = 0; k < kT / 32; ++k)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    umma_f8_warp(tmem + kColO + 48 * j, umma_desc_sw128(sb + j * kCkvBlock + k * 4096, kCkvBlock, 1024),
                                 desc_k(pb + k * 32), kIdescPv, (c | k) != 0);
            umma_commit_warp(bar(bOFull));
            umma_commit_warp(bar(bFree));
            n_pv = g + 1;
            return true;
        };
        bool ok = true;
        int g = 0, n_ne = 0;  // chunks, items with tokens
        for (int j = 0; ok; ++j) {
            const int it = slot_item(a, order, j, n_items);
            if (it >= n_items) break;
            const Item x = item_of(a, it);
            if (x.nch == 0) continue;
            ok = warp_wait(bar(bQFull), n_ne & 1);  // the item's queries are staged
            for (int c = 0; c < x.nch && ok; ++c, ++g) ok = qk(g) && pv(g, c);
            ++n_ne;
        }
        // Every commit's arrival lands before the CTA may exit: wait
        // (bounded) for the newest phase of each barrier committed to.
        if (lane == 0) {
            if (n_qk > 0) (void)mbar_wait_bounded(bar(bSFull), (n_qk - 1) & 1, kWaitLimitNs);
            if (n_pv > 0) {
                (void)mbar_wait_bounded(bar(bOFull), (n_pv - 1) & 1, kWaitLimitNs);
                (void)mbar_wait_bounded(bar(bFree), (n_pv - 1) & 1, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ======================= softmax, epilogue ================================
        const int q = warp & 3;                    // tensor-memory lane quarter
        const int i = threadIdx.x - kWarpSm * 32;  // 0..127
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const float cks = __ldg(a.ckv_scale);
        const float sl = a.scale_log2;
        // The item's queries as FP8 / bf16 B operands (Q8 is free: the last
        // scores that read it are complete), then one arrival per warp.
        // Warp q stages heads 4q .. 4q + 3; lane l holds latent values
        // 8l .. 8l + 7 and 256 + 8l .. 256 + 8l + 7 of each, so every load
        // reads whole 512-byte stretches of a row.
        const bool ql_vec = ((reinterpret_cast<uintptr_t>(a.q_lat) | static_cast<uintptr_t>(a.ql_s0 * 2) |
                              static_cast<uintptr_t>(a.ql_s1 * 2)) & 15) == 0;
        const bool qp_vec = ((reinterpret_cast<uintptr_t>(a.q_pe) | static_cast<uintptr_t>(a.qp_s0 * 2) |
                              static_cast<uintptr_t>(a.qp_s1 * 2)) & 15) == 0;
        auto stage_q = [&](const Item& x) {
            uint4 w[4][2];  // [head][piece]: eight bf16 values each, all loads in flight at once
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                const int h = 4 * q + hh;
                const uint16_t* row = a.q_lat + x.b * a.ql_s0 + h * a.ql_s1 + 8 * lane;
#pragma unroll
                for (int pc = 0; pc < 2; ++pc) {
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (h < H) {
                        if (ql_vec) {
                            v = ldg_nc128(row + 256 * pc);
                        } else {
                            const uint32_t* r32 = reinterpret_cast<const uint32_t*>(row + 256 * pc);
                            v = make_uint4(__ldg(r32), __ldg(r32 + 1), __ldg(r32 + 2), __ldg(r32 + 3));
                        }
                    }
                    w[hh][pc] = v;
                }
            }
            {  // q_pe: lane l holds 16 bytes (part l % 8) of head 4q + l / 8
                const int h = 4 * q + (lane >> 3), p = lane & 7;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (h < H) {
                    const uint16_t* src = a.q_pe + x.b * a.qp_s0 + h * a.qp_s1 + 8 * p;
                    if (qp_vec) {
                        v = ldg_nc128(src);
                    } else {
                        const uint32_t* r32 = reinterpret_cast<const uint32_t*>(src);
                        v = make_uint4(__ldg(r32), __ldg(r32 + 1), __ldg(r32 + 2), __ldg(r32 + 3));
                    }
                }
                sts128u(s0 + kOffQp + h * 128 + ((p ^ (h & 7)) << 4), v.x, v.y, v.z, v.w);
            }
            float qsv[4];
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                const int h = 4 * q + hh;
                float mx = 0.f;
#pragma unroll
                for (int pc = 0; pc < 2; ++pc) {
                    const uint32_t u[4] = {w[hh][pc].x, w[hh][pc].y, w[hh][pc].z, w[hh][pc].w};
#pragma unroll
                    for (int m = 0; m < 4; ++m) mx = fmaxf(mx, fmaxf(fabsf(bf16_lo(u[m])), fabsf(bf16_hi(u[m]))));
                }
                mx = warp_max(mx);
                // 2^k with 2^k mx in (224, 448] (k = 0 for an all-zero head)
                int k = 0;
                if (mx > 0.f) {
                    const int e = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu) - 127;
                    k = min(max(8 - e, -126), 126);
                    if (mx * __uint_as_float(static_cast<uint32_t>(k + 127) << 23) > 448.f) --k;
                }
                const float sc = __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
                qsv[hh] = cks / sc;
                // Two E4M3 terms through f16: every scaled value at or above
                // 2^-17 is exact in f16 and those below round to zero in both
                // terms either way, so the bytes are those of the exact split.
#pragma unroll
                for (int pc = 0; pc < 2; ++pc) {
                    const uint32_t u[4] = {w[hh][pc].x, w[hh][pc].y, w[hh][pc].z, w[hh][pc].w};
                    uint32_t t1[2], t2[2];
#pragma unroll
                    for (int m2 = 0; m2 < 2; ++m2) {
                        uint32_t b1 = 0u, b2 = 0u;
#pragma unroll
                        for (int m = 0; m < 2; ++m) {
                            const uint32_t xw = pack_f16(bf16_lo(u[2 * m2 + m]) * sc, bf16_hi(u[2 * m2 + m]) * sc);
                            const uint32_t e1 = f16x2_to_e4m3x2(xw);
                            const uint32_t e2 = f16x2_to_e4m3x2(hsub2(xw, e4m3x2_to_f16x2(static_cast<uint16_t>(e1))));
                            b1 |= e1 << (16 * m);
                            b2 |= e2 << (16 * m);
                        }
                        t1[m2] = b1;
                        t2[m2] = b2;
                    }
                    // values 256 pc + 8 lane ..: block 2 pc + lane / 16, 16-byte
                    // chunk (lane % 16) / 2, its half lane % 2
                    const int blk = 2 * pc + (lane >> 4), chunk = (lane & 15) >> 1;
                    const uint32_t base = s0 + kOffQ + blk * kQBlock + 8 * (lane & 1);
                    sts64u(base + h * 128 + ((chunk ^ (h & 7)) << 4), t1[0], t1[1]);
                    sts64u(base + (16 + h) * 128 + ((chunk ^ (h & 7)) << 4), t2[0], t2[1]);
                }
            }
            if (lane == 0) sts128(s0 + kOffQs + 16 * q, qsv[0], qsv[1], qsv[2], qsv[3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bQFull));
        };
        // every warp's part of the per-head scales (ckv_scale 2^-k_h) is written
        auto load_qs = [&]() { named_bar_and(1, 128, true); };
        // the slot of the first item with tokens from slot j on (past the
        // end if none); splits without tokens on the way get their
        // (0, -inf) records
        auto next_item = [&](int j) -> int {
            for (;; ++j) {
                const int it = slot_item(a, order, j, n_items);
                if (it >= n_items) return j;
                const Item y = item_of(a, it);
                if (i == 0 && (y.planless || y.plan_bad)) flag_error(a.err, PKV_FLAG_PLAN_RANGE);
                if (y.planless) continue;
                if (i == 0 && y.s == 0 && y.bad_len) flag_error(a.err, PKV_FLAG_SEQ_LEN_RANGE);
                if (y.nch > 0) return j;
                float* op = a.out_partial + y.b * a.op_s0 + y.s * a.op_s1;
                for (int k = i; k < H * kMlaDc; k += 128) op[(k / kMlaDc) * a.op_s2 + (k % kMlaDc)] = 0.f;
                if (i < H) a.lse_partial[y.b * a.lp_s0 + y.s * a.lp_s1 + i] = -INFINITY;
            }
        };

        const int tok = 32 * q + lane;  // token of the chunk = tensor-memory lane
        // The four warps pass the same named barriers and decide whether to
        // go on by the barrier's AND, so all of them stop at the same chunk.
        bool ok = true;
        if (NH < kN) {  // P8 rows of heads NH..15 are never written: P . V reads them as zeros
            for (int k = i; k < kPBytes / 16; k += 128) sts128u(s0 + kOffP + 16 * k, 0u, 0u, 0u, 0u);
        }
        int js = next_item(0);  // schedule slot of the current item
        int it = slot_item(a, order, js, n_items);
        Item x;
        if (it < n_items) {
            x = item_of(a, it);
            stage_q(x);
            load_qs();
        }
        int g = 0;  // chunks of this CTA
        while (it < n_items && ok) {
            float m[NH], l[NH];  // reference maximum (log2 units), this thread's part of the sum
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                m[h] = -INFINITY;
                l[h] = 0.f;
            }
            for (int c = 0; c < x.nch; ++c, ++g) {
                const bool got = warp_wait(bar(bSFull), g & 1);
                const bool live = page_of(x, 2 * c + (tok >> 6), num_pages) >= 0 && tok < x.ntok - kT * c;
                float sv[NH], cm[NH];
                const uint32_t red = s0 + kOffMax;
                if (got) {
                    tc_fence_after();
                    uint32_t r1[NH], r2[NH], rp[NH];
                    const uint32_t ta = tmem + lane_base + kColS;
                    tmem_ld_heads<NH>(ta, r1);
                    tmem_ld_heads<NH>(ta + 16, r2);
                    tmem_ld_heads<NH>(ta + 32, rp);
                    tmem_wait_ld();
#pragma unroll
                    for (int h4 = 0; h4 < NH / 4; ++h4) {
                        const float4 qs = lds128f(s0 + kOffQs + 16 * h4);
                        const float qv[4] = {qs.x, qs.y, qs.z, qs.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int h = 4 * h4 + e;
                            const float lat = __uint_as_float(r1[h]) + __uint_as_float(r2[h]);
                            sv[h] = live ? fmaf(lat, qv[e], __uint_as_float(rp[h])) * sl : -INFINITY;
                            cm[h] = sv[h];
                        }
                    }
#pragma unroll
                    for (int h = 0; h < NH; ++h) cm[h] = warp_max(cm[h]);
                    if (lane == 0)
#pragma unroll
                        for (int h4 = 0; h4 < NH / 4; ++h4)
                            sts128(red + (q * kN + 4 * h4) * 4, cm[4 * h4], cm[4 * h4 + 1], cm[4 * h4 + 2],
                                   cm[4 * h4 + 3]);
                }
                ok = named_bar_and(1, 128, got);
                if (!ok) break;
#pragma unroll
                for (int w = 0; w < 4; ++w)
#pragma unroll
                    for (int h4 = 0; h4 < NH / 4; ++h4) {
                        const float4 y = lds128f(red + (w * kN + 4 * h4) * 4);
                        if (w == 0) {
                            cm[4 * h4] = y.x;
                            cm[4 * h4 + 1] = y.y;
                            cm[4 * h4 + 2] = y.z;
                            cm[4 * h4 + 3] = y.w;
                        } else {
                            cm[4 * h4] = fmaxf(cm[4 * h4], y.x);
                            cm[4 * h4 + 1] = fmaxf(cm[4 * h4 + 1], y.y);
                            cm[4 * h4 + 2] = fmaxf(cm[4 * h4 + 2], y.z);
                            cm[4 * h4 + 3] = fmaxf(cm[4 * h4 + 3], y.w);
                        }
                    }
                // New reference maxima (the same in every thread: the same
                // values and operations). O holds the item's earlier chunks
                // against the old ones; when a finite one moves, O must be
                // scaled before P . V.
                bool scale_o = false;
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    const bool move = cm[h] > m[h] + kRescaleLog2 || (m[h] == -INFINITY && cm[h] > -INFINITY);
                    cm[h] = move ? cm[h] : m[h];  // cm: the new reference
                    scale_o |= move && m[h] > -INFINITY;
                }
                // Chunk g - 1's P . V completed before chunk g's scores (the
                // buffer was free first), so O holds every earlier chunk.
                if (scale_o) {
#pragma unroll 1
                    for (int j = 0; j < 12; ++j) {  // 4 blocks x 3 terms
                        uint32_t r[NH];
                        const uint32_t ta = tmem + lane_base + kColO + 16 * j;
                        tmem_ld_heads<NH>(ta, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int h = 0; h < NH; ++h)
                            r[h] = __float_as_uint(__uint_as_float(r[h]) *
                                                   (m[h] == cm[h] ? 1.f : fast_exp2(m[h] - cm[h])));
                        tmem_st_heads<NH>(ta, r);
                    }
                    tmem_wait_st();
#pragma unroll
                    for (int h = 0; h < NH; ++h) l[h] *= m[h] == cm[h] ? 1.f : fast_exp2(m[h] - cm[h]);
                }
                const uint32_t sb = s0 + kOffSlot;
                if (!live) {  // zero weight: make the ckv row exact zeros for P . V
#pragma unroll
                    for (int blk = 0; blk < 4; ++blk)
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch)  // rotated by token: 8 lanes, 8 bank groups
                            sts128u(sb + blk * kCkvBlock + tok * 128 + (((ch + tok) & 7) << 4), 0u, 0u, 0u, 0u);
                }
                const uint32_t pb = s0 + kOffP;
                const uint32_t colx = static_cast<uint32_t>((tok >> 4) << 4);  // the token's 16-byte chunk, unswizzled
#pragma unroll
                for (int h2 = 0; h2 < NH / 2; ++h2) {
                    float pw[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int h = 2 * h2 + e;
                        const float p = cm[h] == -INFINITY ? 0.f : fast_exp2(sv[h] - cm[h]);
                        l[h] += p;
                        m[h] = cm[h];
                        pw[e] = p * kPScale;
                    }
                    // three E5M2 terms of the pair (head 2 h2 in the low
                    // halves), each rounded to nearest; an E5M2 byte is the
                    // high byte of an f16, so the remainders are f16 and exact
                    const uint32_t xw = pack_f16(pw[0], pw[1]);
                    const uint32_t e1 = f16x2_to_e5m2x2(xw);
                    const uint32_t y = hsub2(xw, prmt(e1, 0u, 0x1404u));
                    const uint32_t e2 = f16x2_to_e5m2x2(y);
                    const uint32_t e3 = f16x2_to_e5m2x2(hsub2(y, prmt(e2, 0u, 0x1404u)));
                    const uint32_t bytes[3][2] = {{e1 & 0xFFu, (e1 >> 8) & 0xFFu},
                                                  {e2 & 0xFFu, (e2 >> 8) & 0xFFu},
                                                  {e3 & 0xFFu, (e3 >> 8) & 0xFFu}};
#pragma unroll
                    for (int t = 0; t < 3; ++t)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int row = 16 * t + 2 * h2 + e;
                            sts8(pb + row * 128 + (colx ^ ((row & 7) << 4)) + (tok & 15), bytes[t][e]);
                        }
                }
                fence_proxy_async_smem();  // P8 and zeroed rows before the tensor core reads them
                tc_fence_before();         // S read and O scaled before the next MMAs
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(bPFull));
            }
            if (!ok) break;
            // The next item's queries first: its scores then overlap this
            // item's epilogue (Q8 is free: this item's last scores are done).
            const int nj = next_item(js + 1);
            const int nxt = slot_item(a, order, nj, n_items);
            Item y;
            if (nxt < n_items) {
                y = item_of(a, nxt);
                stage_q(y);
            }
            // ---- epilogue: l over the tokens of the four warps, O / l ---------------
            const bool got_o = warp_wait(bar(bOFull), (g - 1) & 1);  // the item's last P . V
            // l over the warp's 32 tokens by recursive halving: each step
            // hands half of the heads still held to the partner lane (which
            // keeps the upper half adds n/2 to its head), then the lanes left
            // holding the same head add up; lane 32/NH k ends with head k'.
            float lr[NH];
#pragma unroll
            for (int h = 0; h < NH; ++h) lr[h] = l[h];
            int hl = 0;  // the head this lane ends with
#pragma unroll
            for (int n = NH, off = 16; n > 1; n >>= 1, off >>= 1) {
                const bool up = lane & off;
                hl += up ? n / 2 : 0;
#pragma unroll
                for (int j = 0; j < n / 2; ++j)
                    lr[j] = (up ? lr[j + n / 2] : lr[j]) +
                            __shfl_xor_sync(0xffffffffu, up ? lr[j] : lr[j + n / 2], off);
            }
#pragma unroll
            for (int off = 16 / NH; off >= 1; off >>= 1) lr[0] += __shfl_xor_sync(0xffffffffu, lr[0], off);
            const uint32_t lred = s0 + kOffSum;
            if ((lane & (32 / NH - 1)) == 0)
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(lred + (q * kN + hl) * 4), "f"(lr[0]) : "memory");
            ok = named_bar_and(1, 128, got_o);
            if (!ok) break;
            // Thread h < NH: head h's l over the four warps, its LSE and
            // ckv_scale / (2^7 l) into the (now free) chunk-maxima buffer.
            const uint32_t ired = s0 + kOffMax;
            if (i < NH) {
                float lt = 0.f, mi = -INFINITY;
#pragma unroll
                for (int w = 0; w < 4; ++w) lt += __uint_as_float(lds32(lred + (w * kN + i) * 4));
#pragma unroll
                for (int h = 0; h < NH; ++h) mi = h == i ? m[h] : mi;
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(ired + i * 4),
                             "f"(lt > 0.f ? cks * __frcp_rn(kPScale * lt) : 0.f)
                             : "memory");
                if (i < H)
                    a.lse_partial[x.b * a.lp_s0 + x.s * a.lp_s1 + i] =
                        lt > 0.f ? (mi + __log2f(lt)) * 0.69314718055994530942f : -INFINITY;
            }
            named_bar_and(1, 128, true);
            float inv[NH];
#pragma unroll
            for (int h4 = 0; h4 < NH / 4; ++h4) {
                const float4 v = lds128f(ired + 16 * h4);
                inv[4 * h4] = v.x;
                inv[4 * h4 + 1] = v.y;
                inv[4 * h4 + 2] = v.z;
                inv[4 * h4 + 3] = v.w;
            }
            float* outp = a.out_partial + x.b * a.op_s0 + x.s * a.op_s1;
            tc_fence_after();
#pragma unroll 1
            for (int j2 = 0; j2 < 2; ++j2) {  // two 128-row blocks of O per tensor-memory wait
                uint32_t r[6][NH];
                const uint32_t ta = tmem + lane_base + kColO + 96 * j2;
#pragma unroll
                for (int t = 0; t < 6; ++t) tmem_ld_heads<NH>(ta + 16 * t, r[t]);
                tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                    for (int h = 0; h < NH; ++h)
                        if (h < H)
                            outp[h * a.op_s2 + 128 * (2 * j2 + jj) + 32 * q + lane] =
                                (__uint_as_float(r[3 * jj][h]) + __uint_as_float(r[3 * jj + 1][h]) +
                                 __uint_as_float(r[3 * jj + 2][h])) *
                                inv[h];
            }
            // O is read (waited above) before this warp's next P hand-off,
            // which is what lets the next item's P . V overwrite it.
            tc_fence_before();
            if (nxt < n_items) load_qs();
            it = nxt;
            js = nj;
            x = y;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

int mla_decode_ctas_per_sm(int) { return kCtasPerSm; }

cudaError_t launch_mla_decode(const MlaDecodeArgs& a, const CUtensorMap& tckv, const CUtensorMap& tkpe,
                              cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    // the softmax warps handle 8 heads when there are at most 8, else 16
    auto kernel = a.H <= 8 ? mla_decode_kernel<8> : mla_decode_kernel<16>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
    // persistent: at most two CTAs per SM, each taking one item of every
    // round of gridDim.x schedule positions
    const int64_t items = a.work != nullptr ? a.n_work : static_cast<int64_t>(a.B) * a.num_splits;
    if (items == 0) return cudaSuccess;
    const int grid = static_cast<int>(std::min<int64_t>(items, static_cast<int64_t>(kCtasPerSm) * sms));
    return launch_dependent(kernel, dim3(grid), dim3(kThreads), kSmem, s, tckv, tkpe, a);
}

}  // namespace pkv
