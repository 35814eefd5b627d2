// pa_prefix.cuh -- chunked-prefix (prefill) attention over the paged cache on the sm_103a
// tensor cores (tcgen05, accumulators in tensor memory).  "paged_attn.py", forward_prefix /
// _forward_prefix_pytorch.
//
// Sequence s has ctx = context_lens[s] tokens in the paged cache and q_len new tokens whose
// query/key/value rows are dense (rows query_start_loc[s] .. query_start_loc[s+1]-1).  New
// token j of query head h sees every context token (no mask) and new tokens 0..j (causal),
// through kv head h / G:  out = softmax(scale * q K^T) V.
//
// One CTA owns (sequence, kv head, 128 query rows), a row being a (new token j, head g of
// the kv head's group) pair numbered j * G + g: every key/value tile is read once per kv head
// and shared by the whole GQA group, and the 128 rows are the M of every MMA.  Tiles of 64
// keys; ten warps with fixed roles:
//   key / value loader warps (two each) fill separate rings of key and value slots in shared
//                  memory, in the canonical K-major layouts: keys as [key/8][d/8][8 keys][8]
//                  (no swizzle), values as whole pages [d][block_size keys] with the 32- or
//                  64-byte swizzle (block size 16 / 32; plain rows for 8).  A tile of full,
//                  valid pages moves by tensor copies (TMA), one lane per key box (8 tokens,
//                  128-byte rows) or value page; the context's last tile, a tile with a page
//                  outside the cache, and the chunk's dense rows move by 16-byte cp.async
//                  (zero-filling what must not count; dense value rows transposed on the way).
//                  A key slot is free once its score MMA is done, a value slot only after the
//                  value MMA, so the key ring runs further ahead.
//   score-MMA lane S = Q K^T (M 128, N 64, Q in tensor memory) into one of two S buffers.
//                  Where tensor memory cannot hold two S buffers next to O, Q and P (head
//                  size 256, 192 in bf16), the second half of Q is read from shared memory.
//   value-MMA lane O += P V (N = head size, P in tensor memory where it fits, else in shared
//                  memory) once the softmax has written P.  An MMA issue blocks the issuing
//                  thread until the tensor core takes it, so the two products have a lane each.
//   softmax warps  one thread per row: read the row of S from tensor memory, mask, exp2 with
//                  a running reference max that only moves when the row max grows by more
//                  than 2^8 (then O and the row sum are rescaled), write P (bf16 as hi + lo
//                  so probabilities keep ~16 bits) in the value MMA's A layout.
// All waits are bounded (about two seconds); a wait that gives up sets an abort flag every
// role checks and bit 2 of the device error word, and the CTA still drains its MMAs and frees
// its tensor memory before it exits.
#pragma once

#include "pa_kernels.cuh"
#include "pa_prefix.h"
#include "pa_tc.cuh"

// Tuning knobs (compile-time): PA_PFX_QSPLIT lets the second half of Q live in shared memory
// where that buys a second S buffer; PA_PFX_KEY_SHARE is the key ring's share of the
// key/value slots, in eighths; PA_PFX_WAIT_HINT_NS is the suspend hint of the bounded waits.
#ifndef PA_PFX_QSPLIT
#define PA_PFX_QSPLIT 1
#endif
#ifndef PA_PFX_KEY_SHARE
#define PA_PFX_KEY_SHARE 4
#endif
#ifndef PA_PFX_WAIT_HINT_NS
#define PA_PFX_WAIT_HINT_NS 20000
#endif

namespace pa {

template <bool BF16, int D>
struct PfxCfg {
    static constexpr int DP = (D + 15) / 16 * 16;  // head size padded to the MMA K step
    static constexpr int DPR = (DP + 31) / 32 * 32;  // O columns read in 32-column pieces
    static constexpr int NCR = D / 8;              // 16-byte chunks of a row that exist
    static constexpr int NCP = DP / 8;             // chunks after padding
    static constexpr int BN = 64;                  // keys per tile
    static constexpr int NP = BF16 ? 2 : 1;        // P terms: hi (and lo for bf16)
    static constexpr int K_BYTES = BN * DP * 2;    // a key tile; a value tile is as large
    static constexpr int V_BYTES = BN * DP * 2;
    static constexpr int P_BYTES = kPfxBM * BN * 2;
    static constexpr int CTL_BYTES = 512;
    // Tensor memory: S buffers, O, Q and (where they fit) the two P buffers, the A operand of
    // the value MMA.  Two S buffers with P in tensor memory; else the same with half of Q in
    // shared memory; else one S buffer with P in tensor memory; else two S buffers with P in
    // shared memory.
    static constexpr int TM_OQ = DPR + DP / 2, TM_P = 2 * NP * (BN / 2);
    static constexpr bool FIT2 = 2 * BN + TM_OQ + TM_P <= 512;
    // Where two S buffers do not fit, keeping the second half of Q in shared memory (the
    // score MMA's A operand for the last DP / 32 K steps) may make them fit.
    static constexpr bool QSPLIT = !FIT2 && PA_PFX_QSPLIT && 2 * BN + DPR + DP / 4 + TM_P <= 512;
    static constexpr bool FIT1 = BN + TM_OQ + TM_P <= 512;
    static constexpr bool P_TMEM = FIT2 || QSPLIT || FIT1;
    static constexpr int NSB = (FIT2 || QSPLIT) ? 2 : (FIT1 ? 1 : 2);  // S buffers
    static constexpr int P_SMEM = P_TMEM ? 0 : 2 * NP * P_BYTES;
    static constexpr int QT = QSPLIT ? DP / 2 : DP;  // head elements of Q in tensor memory
    static constexpr int Q_SMEM = QSPLIT ? kPfxBM * (DP - QT) * 2 : 0;
    // Separate key and value rings: a key slot is free once the score MMA (and the softmax's
    // look at the tile's masks) is done, a value slot only after the value MMA.
    static constexpr int SLOTS = (227 * 1024 - P_SMEM - Q_SMEM - CTL_BYTES) / K_BYTES;
    static constexpr int NK0 = SLOTS * PA_PFX_KEY_SHARE / 8;  // key share of the slots (in eighths)
    static constexpr int NK = NK0 > 8 ? 8 : (NK0 < 2 ? 2 : NK0);
    static constexpr int NV = SLOTS - NK > 8 ? 8 : SLOTS - NK;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = NK * K_BYTES;
    static constexpr int OFF_P = OFF_V + NV * V_BYTES;
    static constexpr int OFF_Q = OFF_P + P_SMEM;  // [chunk][128 rows][16 bytes] of Q's second half
    static constexpr int OFF_CTL = OFF_Q + Q_SMEM;
    // at least 120 KiB so two CTAs never share an SM (each takes all 512 tensor-memory columns)
    static constexpr int SMEM = OFF_CTL + CTL_BYTES > 120 * 1024 ? OFF_CTL + CTL_BYTES : 120 * 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0;                 // S buffer b: [b BN, (b + 1) BN)
    static constexpr uint32_t COL_O = NSB * BN;          // O: [COL_O, COL_O + DPR)
    static constexpr uint32_t COL_Q = COL_O + DPR;       // Q, two 16-bit values per column: DP / 2
    static constexpr uint32_t COL_P = COL_Q + QT / 2;    // P buffer b, term h: + (b NP + h) BN / 2
    static constexpr uint32_t IDESC_S = umma_idesc_f16(BF16, kPfxBM, BN);
    static constexpr uint32_t IDESC_O = umma_idesc_f16(BF16, kPfxBM, DP);
    static_assert(COL_Q + QT / 2 <= TMEM_COLS, "tensor memory");
    static_assert(!P_TMEM || COL_P + TM_P <= TMEM_COLS, "tensor memory");
    static_assert(NV >= 2 && SMEM <= 227 * 1024, "shared memory");
};

static __device__ unsigned int g_prefix_errors = 0;

__device__ __forceinline__ void prefix_flag(unsigned int bit) { atomicOr(&g_prefix_errors, bit); }

// Bounded wait on an mbarrier phase; gives up when another role has aborted or after the
// wait limit (then it raises the abort flag itself).
__device__ __forceinline__ bool pfx_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_hint(bar, parity, PA_PFX_WAIT_HINT_NS)) {
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            prefix_flag(4u);
            return false;
        }
    }
    return true;
}

// Byte offset of (token o of a tile, value row dd) in a value tile.  The tile is pages of
// block_size keys, DP * 2 * block_size bytes apart; a page is DP rows of 2 * block_size bytes
// whose 16-byte chunks are XOR-swizzled the way the value MMA reads them (none for block
// size 8, row bit 2 for 16 = 32-byte swizzle, row bits 1-2 for 32 = 64-byte swizzle), which
// is also what a swizzled tensor copy of a whole page writes.
__device__ __forceinline__ uint32_t pfx_v_off(int o, int dd, int bs_log2, int DP) {
    const int rowb_log2 = bs_log2 + 1;
    const int kq = (o >> 3) & ((1 << (bs_log2 - 3)) - 1);
    const int swz = bs_log2 == 3 ? 0 : (bs_log2 == 4 ? (dd >> 2) & 1 : (dd >> 1) & 3);
    return (uint32_t)((o >> bs_log2) * (DP << rowb_log2) + (dd << rowb_log2) + ((kq ^ swz) << 4));
}

// How a sequence's n_ctx context tiles are split: {number of splits, tiles per split}.  A
// context longer than split_tiles tiles is cut into at most nsplit equal parts; every split
// holds at least one tile, the last one also takes the chunk.
__device__ __forceinline__ int2 pfx_split_plan(int n_ctx, int nsplit, int split_tiles) {
    int ns = n_ctx > split_tiles ? min(nsplit, (n_ctx + split_tiles - 1) / split_tiles) : 1;
    const int per = max(1, (n_ctx + ns - 1) / ns);
    ns = max(1, (n_ctx + per - 1) / per);
    return make_int2(ns, per);
}

// Sequence order of the grid's z: sequences sorted by the work of one of their CTAs (its
// context part plus the chunk tiles of its heaviest row tile), largest first, ties by index.
// The hardware hands out CTAs roughly in grid order, so long CTAs start first and short ones
// fill the end of the grid instead of long ones trailing behind.  Every CTA ranks all
// sequences itself (one parallel load per sequence and a rank count; no workspace, no extra
// launch); above kPfxOrderSeqs sequences the grid order stands.  Called by every thread at
// kernel entry; `scratch` holds kPfxOrderSeqs + 1 words of shared memory, free afterwards.
constexpr int kPfxOrderSeqs = 120;
__device__ __forceinline__ int pfx_seq_order(const PrefixParams& p, int z, uint32_t* scratch) {
    const int S = gridDim.z;
    if (S == 1 || S > kPfxOrderSeqs) return z;
    for (int t = threadIdx.x; t < S; t += blockDim.x) {
        int c = p.ctx_lens[t];
        const int q = p.qsl[t + 1] - p.qsl[t];
        uint32_t w = 0;
        if (c >= 0 && q >= 0 && q <= p.max_query_len) {
            c = min(c, p.mbps * p.bs);
            const int n = (c + 63) / 64;
            const int2 plan = pfx_split_plan(n, p.nsplit, p.split_tiles);
            w = (uint32_t)(min(plan.y, n) + (q + 63) / 64);
        }
        scratch[t] = w;
    }
    __syncthreads();
    for (int t = threadIdx.x; t < S; t += blockDim.x) {
        const uint32_t w = scratch[t];
        int r = 0;
        for (int j = 0; j < S; ++j) {
            const uint32_t wj = scratch[j];
            r += (wj > w || (wj == w && j < t)) ? 1 : 0;
        }
        if (r == z) scratch[kPfxOrderSeqs] = (uint32_t)t;
    }
    __syncthreads();
    const int s = (int)scratch[kPfxOrderSeqs];
    __syncthreads();
    return s;
}

// One lane waits, the warp learns the outcome (warp-uniform, as tcgen05.ld/st require).
__device__ __forceinline__ bool pfx_warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int lane) {
    int ok = 1;
    if (lane == 0) ok = pfx_wait(bar, parity, abort_flag);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
}

// Zero the slot bytes the copies never write: key chunks c >= D/8 of every key slot, value
// rows d >= D of every value slot (the MMAs read the head size padded to 16).
template <class C, int D>
__device__ __forceinline__ void pfx_zero_padding(uint8_t* smem, const PrefixParams& p, int tid, int nthreads) {
    constexpr int BN = C::BN, NK = C::NK, NV = C::NV;
    if constexpr (C::NCP > C::NCR) {
        constexpr int kpad = (C::NCP - C::NCR) * BN, vpad = (BN / 8) * (C::DP - D);
        for (int i = tid; i < NK * kpad + NV * vpad; i += nthreads) {
            uint8_t* dst;
            if (i < NK * kpad) {
                const int slot = i / kpad, rem = i % kpad;
                const int o = rem % BN, c = C::NCR + rem / BN;
                dst = smem + C::OFF_K + slot * C::K_BYTES + (o >> 3) * (C::DP * 16) + c * 128 + (o & 7) * 16;
            } else {
                const int j = i - NK * kpad, slot = j / vpad, rem = j % vpad;
                const int kc = rem / (C::DP - D), dd = D + rem % (C::DP - D);
                const int cpp_log2 = p.bs_log2 - 3;  // 16-byte chunks per value row, log2
                dst = smem + C::OFF_V + slot * C::V_BYTES + (kc >> cpp_log2) * (C::DP << (p.bs_log2 + 1)) +
                      (dd << (p.bs_log2 + 1)) + ((kc & ((1 << cpp_log2) - 1)) << 4);
            }
            *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// The key range one CTA attends: context tiles [tb, tb + n_ctx) of a sequence with ctx cached
// tokens (context tile i holds tokens 64 i ..), then, in the sequence's last split, the chunk's
// tiles; n_tiles in all.  Chunk rows are q0 .. q0 + q_len - 1 of key/value.
struct PfxRange {
    int tb, n_ctx, ctx, n_tiles, q0, q_len, kvh;
    const int32_t* table;  // the sequence's block-table row
};

// Loader role of the prefix kernels: a team of TEAM threads (whole warps; lanes of the first
// warp issue the tensor copies) fills the key ring (kteam) or the value ring of the layout C.
// lt = thread index in the team.
template <class C, int D, int TEAM>
__device__ __forceinline__ void pfx_load_tiles(const PrefixParams& p, const PfxRange& g, bool kteam, int lt, int lane,
                                               uint32_t sbase, uint64_t* k_full, uint64_t* k_empty, uint64_t* v_full,
                                               uint64_t* v_empty, uint32_t* bad_mask, volatile int* abort_flag) {
    constexpr int BN = C::BN, NK = C::NK, NV = C::NV;
    const int tb = g.tb, n_ctx = g.n_ctx, ctx = g.ctx, n_tiles = g.n_tiles, q0 = g.q0, q_len = g.q_len, kvh = g.kvh;
    const int32_t* table = g.table;
    const int64_t page_bytes = (int64_t)D * p.bs * 2;
    const int npg = BN >> p.bs_log2;  // pages per context tile
    // lane i < npg holds the block id of page i of a context tile (-1 past the context);
    // the ids of tile t + 1 are loaded while tile t is waited for and issued
    auto tile_page = [&](int t) {
        int b = -1;
        if (t < n_ctx && lane < npg && (tb + t) * BN + (lane << p.bs_log2) < ctx)
            b = table[(((tb + t) * BN) >> p.bs_log2) + lane];
        return b;
    };
    int pid_next = tile_page(0);
    int t = 0;
    for (; t < n_tiles; ++t) {
        const int pid = pid_next;
        pid_next = tile_page(t + 1);
        const int slot = kteam ? t % NK : t % NV;
        uint64_t* full = kteam ? &k_full[slot] : &v_full[slot];
        if (kteam ? t >= NK : t >= NV) {
            if (!pfx_warp_wait(kteam ? &k_empty[slot] : &v_empty[slot], ((t / (kteam ? NK : NV)) - 1) & 1,
                               abort_flag, lane))
                break;
        }
        const uint32_t sK = sbase + C::OFF_K + slot * C::K_BYTES;
        const uint32_t sV = sbase + C::OFF_V + slot * C::V_BYTES;
        bool generic = true;  // this warp wrote the slot through the generic proxy (cp.async / st.shared)
        if (t < n_ctx) {
            const int t0 = (tb + t) * BN;
            // pages of the tile whose id is outside the cache (masked); both teams compute
            // the same mask
            const bool bad = lane < npg && t0 + (lane << p.bs_log2) < ctx && (unsigned)pid >= (unsigned)p.num_blocks;
            const uint32_t m = __ballot_sync(0xffffffffu, bad);
            const bool tma = m == 0 && t0 + BN <= ctx;  // a full tile of valid pages
            generic = !tma;
            if (lt < 32) {
                if (lane == 0) {
                    if (kteam) {
                        bad_mask[slot] = m;
                        if (m) prefix_flag(32u);
                    }
                    if (tma)
                        mbar_arrive_expect_tx(full, 2u * BN * D);
                    else
                        mbar_arrive(full);
                }
                __syncwarp();
                if (tma && kteam) {
                    // keys: tensor copies of 128-byte rows, one box of 8 tokens per lane
                    const int kpage = __shfl_sync(0xffffffffu, pid, (8 * lane) >> p.bs_log2 & 31) * p.Hk + kvh;
                    if (lane < BN / 8)
                        tma_load_4d(sK + lane * (C::DP * 16), &p.kmap, 0, ((8 * lane) & (p.bs - 1)) >> 3, 0, kpage,
                                    full);
                } else if (tma && lane < npg) {
                    // values: one whole page per lane, swizzled as the value MMA reads it
                    const int vpage = pid * p.Hk + kvh;
                    const uint32_t dst = sV + lane * (C::DP << (p.bs_log2 + 1));
                    if (p.bs_log2 == 3)
                        bulk_load(dst, p.vcache + (int64_t)vpage * page_bytes, (uint32_t)page_bytes, full);
                    else
                        tma_load_3d(dst, &p.vmap, 0, 0, vpage, full);
                }
            }
            if (!tma && kteam) {
                // keys of the context's last tile or of a tile with a page outside the cache:
                // 16-byte pieces, past the context or of a masked page zero-filled
                const int kper = C::NCR << p.bs_log2;
                for (int base = 0; base < BN * C::NCR; base += TEAM) {
                    const int i = base + lt;
                    const bool act = i < BN * C::NCR;
                    const int pg = act ? i / kper : 0, rem = i - pg * kper;
                    const int b = __shfl_sync(0xffffffffu, pid, pg);
                    if (act) {
                        const int c = rem >> p.bs_log2, sl = rem & (p.bs - 1);
                        const int o = (pg << p.bs_log2) + sl;
                        const bool ok = t0 + o < ctx && (unsigned)b < (unsigned)p.num_blocks;
                        const uint8_t* src = ok ? p.kcache + ((int64_t)b * p.Hk + kvh) * page_bytes +
                                                      (int64_t)(c * p.bs + sl) * 16
                                                : p.kcache;
                        cp_async16(sK + (o >> 3) * (C::DP * 16) + c * 128 + (o & 7) * 16, src, ok ? 16u : 0u);
                    }
                }
            } else if (!tma) {
                // values: 8-key pieces of each page row; the part past the context or of a
                // masked page reads as zero
                const int kpp_log2 = p.bs_log2 - 3;
                const int vper = D << kpp_log2;
                for (int base = 0; base < (BN / 8) * D; base += TEAM) {
                    const int i = base + lt;
                    const bool act = i < (BN / 8) * D;
                    const int pg = act ? i / vper : 0, rem = i - pg * vper;
                    const int b = __shfl_sync(0xffffffffu, pid, pg);
                    if (act) {
                        const int dd = rem >> kpp_log2, kq = rem & ((1 << kpp_log2) - 1);
                        const int o = (pg << p.bs_log2) + kq * 8;
                        const int nv = min(max(ctx - t0 - o, 0), 8);
                        const bool ok = nv > 0 && (unsigned)b < (unsigned)p.num_blocks;
                        const uint8_t* src = ok ? p.vcache + ((int64_t)b * p.Hk + kvh) * page_bytes +
                                                      ((int64_t)dd * p.bs + kq * 8) * 2
                                                : p.vcache;
                        cp_async16(sV + pfx_v_off(o, dd, p.bs_log2, C::DP), src, ok ? (uint32_t)nv * 2u : 0u);
                    }
                }
            }
        } else {
            const int kc0 = (t - n_ctx) * BN;
            if (lt == 0) mbar_arrive(full);  // no tensor copies for chunk tiles
            if (kteam) {
                for (int i = lt; i < BN * C::NCR; i += TEAM) {
                    const int c = i / BN, o = i % BN;
                    const int j = kc0 + o;
                    const bool ok = j < q_len;
                    const uint8_t* src =
                        ok ? p.k + ((int64_t)(q0 + j) * p.kv_stride + (int64_t)kvh * D + c * 8) * 2 : p.k;
                    cp_async16(sK + (o >> 3) * (C::DP * 16) + c * 128 + (o & 7) * 16, src, ok ? 16u : 0u);
                }
            } else {
                // dense value rows, two tokens at a time, transposed into the value layout;
                // the loads of four such pieces are in flight together
                constexpr int ITEMS = (BN / 2) * C::NCR, BATCH = 4;
                for (int i0 = 0; i0 < ITEMS; i0 += TEAM * BATCH) {
                    uint4 a[BATCH], b[BATCH];
#pragma unroll
                    for (int u = 0; u < BATCH; ++u) {
                        const int i = i0 + u * TEAM + lt;
                        const int c = i % C::NCR, t2 = 2 * (i / C::NCR), j = kc0 + t2;
                        const uint8_t* vb = p.v + ((int64_t)kvh * D + c * 8) * 2;
                        a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
                        if (i < ITEMS && j < q_len) a[u] = ld_nc_v4(vb + (int64_t)(q0 + j) * p.kv_stride * 2);
                        if (i < ITEMS && j + 1 < q_len) b[u] = ld_nc_v4(vb + (int64_t)(q0 + j + 1) * p.kv_stride * 2);
                    }
#pragma unroll
                    for (int u = 0; u < BATCH; ++u) {
                        const int i = i0 + u * TEAM + lt;
                        if (i >= ITEMS) continue;
                        const int c = i % C::NCR, t2 = 2 * (i / C::NCR);
                        const uint32_t av[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
                        const uint32_t bv[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            sts_u32(sV + pfx_v_off(t2, c * 8 + e, p.bs_log2, C::DP) + (t2 & 7) * 2,
                                    __byte_perm(av[e >> 1], bv[e >> 1], (e & 1) ? 0x7632 : 0x5410));
                    }
                }
            }
        }
        if (generic) {  // make those writes visible to the tensor core before the arrive
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(full);
    }
    cp_async_wait<0>();
    if (t < n_tiles && lt == 0) {
        // Aborted: tensor copies this team issued for its last tiles may still be landing in
        // shared memory.  Wait (bounded) until each slot's latest fill is complete, so that
        // no copy outlives the CTA.
        const int ns = kteam ? NK : NV;
        for (int u = t > ns ? t - ns : 0; u < t; ++u)
            (void)mbar_wait_bounded(kteam ? &k_full[u % ns] : &v_full[u % ns], (uint32_t)(u / ns) & 1u, kWaitLimitNs);
    }
}

template <bool BF16, int D>
__global__ void __launch_bounds__(kPfxThreads, 1) pa_prefix_kernel(const __grid_constant__ PrefixParams p) {
    using C = PfxCfg<BF16, D>;
    constexpr int BN = C::BN, NK = C::NK, NV = C::NV, NSB = C::NSB;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = pfx_seq_order(p, blockIdx.z, reinterpret_cast<uint32_t*>(smem + C::OFF_CTL)), kvh = blockIdx.y;
    const int split = blockIdx.x / p.mt;                        // which part of the context
    const int row0 = (p.mt - 1 - blockIdx.x % p.mt) * kPfxBM;  // row tiles with more keys first
    const int G = p.G;
    int ctx = p.ctx_lens[s];
    const int q0 = p.qsl[s];
    const int q_len = p.qsl[s + 1] - q0;
    if (q_len < 0 || q_len > p.max_query_len || ctx < 0) {
        if (tid == 0 && split == 0) prefix_flag(128u);
        return;
    }
    const int rows_total = q_len * G;
    if (row0 >= rows_total) return;
    if (ctx > p.mbps * p.bs) {  // the table cannot hold the context: cap it (and report)
        if (tid == 0) prefix_flag(64u);
        ctx = p.mbps * p.bs;
    }
    // This CTA's keys: context tiles [tb, tb + n_ctx) of `split`, and the chunk if it is the
    // sequence's last split.
    const int2 plan = pfx_split_plan((ctx + BN - 1) / BN, p.nsplit, p.split_tiles);
    if (split >= plan.x) return;
    const int tb = split * plan.y;
    const int n_ctx = min(plan.y, (ctx + BN - 1) / BN - tb);
    const bool last_split = split == plan.x - 1;

    const uint32_t sbase = smem_addr(smem);
    if (sbase & 1023u) {  // the swizzled layouts are defined on 1 KiB-aligned addresses
        if (tid == 0) prefix_flag(4u);
        return;
    }
    uint8_t* ctl = smem + C::OFF_CTL;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ctl);
    uint64_t* k_full = bars;                 // [NK] keys (and the tile's page mask) in place
    uint64_t* k_empty = k_full + NK;         // [NK] score MMA done and masks read
    uint64_t* v_full = k_empty + NK;         // [NV] values in place
    uint64_t* v_empty = v_full + NV;         // [NV] value MMA done
    uint64_t* s_full = v_empty + NV;         // [NSB]
    uint64_t* s_empty = s_full + NSB;        // [NSB]
    uint64_t* q_full = s_empty + NSB;
    // [2] each: P of even / odd tiles written, value MMAs of even / odd tiles done.  One
    // barrier per P buffer: the softmax reaches tile t's arrive only after tile t-2's value
    // MMA completed, so no barrier ever runs two phases ahead of its waiter.
    uint64_t* p_full = q_full + 1;
    uint64_t* o_done = p_full + 2;
    uint64_t* fin = o_done + 2;  // [2]: every score / value MMA issued has completed
    constexpr int NBARS = 2 * NK + 2 * NV + 2 * NSB + 7;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl + 8 * NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(ctl + 8 * NBARS + 4);
    uint32_t* bad_mask = reinterpret_cast<uint32_t*>(ctl + 8 * NBARS + 8);  // [NK] pages outside the cache
    static_assert(8 * NBARS + 8 + 4 * NK <= C::CTL_BYTES, "control block");
    static_assert(4 * (kPfxOrderSeqs + 1) <= C::CTL_BYTES, "sequence-order scratch");

    const int row_last = min(row0 + kPfxBM, rows_total) - 1;
    const int n_tiles = n_ctx + (last_split ? (row_last / G) / BN + 1 : 0);

    if (tid == 0) {
        for (int i = 0; i < NK; ++i) {
            mbar_init(&k_full[i], 3);   // the key-copy arrive (+ bytes) and the two key warps
            mbar_init(&k_empty[i], 5);  // the score MMA's commit and the four softmax warps
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&v_full[i], 3);   // the value-copy arrive (+ bytes) and the two value warps
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < NSB; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 4);
        }
        mbar_init(q_full, 4);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&p_full[i], 4);
            mbar_init(&o_done[i], 1);
            mbar_init(&fin[i], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    pfx_zero_padding<C, D>(smem, p, tid, kPfxThreads);
    fence_proxy_async_smem();
    if (warp == kPfxMmaWarp) tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tmem_slot;
    const int32_t* table = p.block_tables + (int64_t)s * p.mbps;
    const PfxRange rng{tb, n_ctx, ctx, n_tiles, q0, q_len, kvh, table};
    const bool kteam = warp >= kPfxKeyWarp0 && warp < kPfxKeyWarp0 + 2;
    const bool vteam = warp >= kPfxValWarp0 && warp < kPfxValWarp0 + 2;
    if (kteam || vteam) {
        // ------------------------------------------------------------------ loaders
        // two warps fill the key ring, two the value ring; each team runs on its own
        const int lt = tid - (kteam ? kPfxKeyWarp0 : kPfxValWarp0) * 32;  // 0 .. 63 in the team
        pfx_load_tiles<C, D, 64>(p, rng, kteam, lt, lane, sbase, k_full, k_empty, v_full, v_empty, bad_mask,
                                 abort_flag);
    } else if (warp == kPfxMmaWarp) {
        // ------------------------------------------------------------------ score MMAs
        if (lane == 0) {
            // S of tile t as soon as its keys are in and the softmax has read S of tile
            // t - NSB out of the same buffer
            // Descriptors as a constant high half and a low half that is the start address
            // (>> 4) plus the layout's fixed low bits: one add per MMA.  A lane that shares its
            // sub-partition with a softmax warp gets few issue slots while that warp runs a
            // dense stretch of arithmetic, so every instruction saved here shortens the chain.
            const uint64_t kd0 = umma_desc(sbase + C::OFF_K, 128, C::DP * 16);
            const uint32_t kd_lo = (uint32_t)kd0, kd_hi = (uint32_t)(kd0 >> 32);
            const uint64_t qd0 = umma_desc(sbase + C::OFF_Q, kPfxBM * 16, 128);
            const uint32_t qd_lo = (uint32_t)qd0, qd_hi = (uint32_t)(qd0 >> 32);
            bool ok = pfx_wait(q_full, 0, abort_flag);
            for (int t = 0; ok && t < n_tiles; ++t) {
                ok = pfx_wait(&k_full[t % NK], (t / NK) & 1, abort_flag) &&
                     (t < NSB || pfx_wait(&s_empty[t % NSB], ((t / NSB) - 1) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                const uint32_t k_lo = kd_lo + (uint32_t)((t % NK) * (C::K_BYTES >> 4));
                const uint32_t d_s = tm + C::COL_S + (t % NSB) * BN;
#pragma unroll
                for (int ks = 0; ks < C::DP / 16; ++ks) {
                    // K step ks: 16 head elements = two 128-byte chunk columns of the key tile
                    if (ks < C::QT / 16)
                        umma_f16_ts(d_s, tm + C::COL_Q + ks * 8, k_lo + ks * 16, kd_hi, C::IDESC_S, ks > 0 ? 1u : 0u);
                    else
                        umma_f16_ss(d_s, qd_lo + (ks - C::QT / 16) * (2 * kPfxBM), qd_hi, k_lo + ks * 16, kd_hi,
                                    C::IDESC_S, 1u);
                }
                umma_commit(&s_full[t % NSB]);
                umma_commit(&k_empty[t % NK]);
            }
            // every MMA issued has completed before tensor memory is released
            umma_commit(&fin[0]);
            if (!mbar_wait_bounded(&fin[0], 0, kWaitLimitNs)) prefix_flag(4u);
        }
        __syncwarp();
    } else if (warp == kPfxPvWarp) {
        // ------------------------------------------------------------------ value MMAs
        if (lane == 0) {
            // value-tile descriptor: the block size fixes the layout; 16 keys (one K step) are
            // two 8-row pages (block size 8), one page with the 32-byte swizzle (16) or half a
            // page with the 64-byte swizzle (32), at these byte offsets in the tile
            const uint64_t vd0 = p.bs_log2 == 3   ? umma_desc(sbase + C::OFF_V, C::DP * 16, 128)
                                 : p.bs_log2 == 4 ? umma_desc_sw(sbase + C::OFF_V, 256, 6)
                                                  : umma_desc_sw(sbase + C::OFF_V, 512, 4);
            const uint32_t vd_lo = (uint32_t)vd0, vd_hi = (uint32_t)(vd0 >> 32);
            uint32_t voff[BN / 16];
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
                voff[kk] = (uint32_t)(p.bs_log2 == 3   ? kk * 2 * (C::DP * 16)
                                      : p.bs_log2 == 4 ? kk * (C::DP * 32)
                                                       : (kk >> 1) * (C::DP * 64) + (kk & 1) * 32) >> 4;
            const uint64_t pd0 = umma_desc(sbase + C::OFF_P, kPfxBM * 16, 128);
            const uint32_t pd_lo = (uint32_t)pd0, pd_hi = (uint32_t)(pd0 >> 32);
            bool ok = true;
            for (int t = 0; ok && t < n_tiles; ++t) {
                ok = pfx_wait(&p_full[t & 1], (t >> 1) & 1, abort_flag) && pfx_wait(&v_full[t % NV], (t / NV) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                const uint32_t v_lo = vd_lo + (uint32_t)((t % NV) * (C::V_BYTES >> 4));
                const uint32_t acc0 = t > 0 ? 1u : 0u;
#pragma unroll
                for (int h = 0; h < C::NP; ++h)
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        const uint32_t acc = (kk > 0 || h > 0) ? 1u : acc0;
                        if constexpr (C::P_TMEM)
                            umma_f16_ts(tm + C::COL_O, tm + C::COL_P + ((t & 1) * C::NP + h) * (BN / 2) + kk * 8,
                                        v_lo + voff[kk], vd_hi, C::IDESC_O, acc);
                        else
                            umma_f16_ss(tm + C::COL_O,
                                        pd_lo + (((t & 1) * C::NP + h) * C::P_BYTES + kk * 2 * (kPfxBM * 16)) / 16, pd_hi,
                                        v_lo + voff[kk], vd_hi, C::IDESC_O, acc);
                    }
                umma_commit(&o_done[t & 1]);
                umma_commit(&v_empty[t % NV]);
            }
            umma_commit(&fin[1]);
            if (!mbar_wait_bounded(&fin[1], 0, kWaitLimitNs)) prefix_flag(4u);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ softmax
        const int sw = warp - kPfxSoftmaxWarp0;  // = warp % 4: this warp's tensor-memory lane quarter
        const int r = sw * 32 + lane;
        const int row = row0 + r;
        const int lim = row / G;  // newest chunk key this row sees (rows past the chunk are never stored)
        const uint32_t tl = tm + ((uint32_t)(sw * 32) << 16);
        const uint32_t sP0 = sbase + C::OFF_P + r * 16;
        // this thread's query row into tensor memory (two 16-bit values per column; rows past
        // the chunk and the padding past D are zero)
        {
            const uint8_t* qrow = nullptr;
            if (row < rows_total) {
                const int j = row / G, g = row - j * G;
                qrow = p.q + ((int64_t)(q0 + j) * p.q_stride + (int64_t)(kvh * G + g) * D) * 2;
            }
#pragma unroll 1
            for (int c = 0; c < C::QT / 16; ++c) {
                uint4 a = make_uint4(0u, 0u, 0u, 0u), b = make_uint4(0u, 0u, 0u, 0u);
                if (qrow != nullptr && 2 * c < C::NCR) a = ld_nc_v4(qrow + c * 32);
                if (qrow != nullptr && 2 * c + 1 < C::NCR) b = ld_nc_v4(qrow + c * 32 + 16);
                const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                                 tl + C::COL_Q + c * 8),
                             "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                             : "memory");
            }
            if constexpr (C::QSPLIT) {
                // the second half as 16-byte chunks [chunk][row] (the score MMA's no-swizzle
                // K-major A layout); the padding past D is zero
                for (int c = C::QT / 8; c < C::NCP; ++c) {
                    uint4 a = make_uint4(0u, 0u, 0u, 0u);
                    if (qrow != nullptr && c < C::NCR) a = ld_nc_v4(qrow + c * 16);
                    sts_v4(sbase + C::OFF_Q + (c - C::QT / 8) * (kPfxBM * 16) + r * 16, a.x, a.y, a.z, a.w);
                }
                fence_proxy_async_smem();
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_full);
        }
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int t = 0; t < n_tiles; ++t) {
            const int ks = t % NK;
            ok = pfx_warp_wait(&k_full[ks], (t / NK) & 1, abort_flag, lane) &&
                 pfx_warp_wait(&s_full[t % NSB], (t / NSB) & 1, abort_flag, lane);
            if (!ok) break;
            tc_fence_after();
            float sv[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c)
                tmem_ld32(tl + C::COL_S + (t % NSB) * BN + c * 32, *reinterpret_cast<float(*)[32]>(&sv[c * 32]));
            const uint32_t bad = t < n_ctx ? bad_mask[ks] : 0u;
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&s_empty[t % NSB]);
                mbar_arrive(&k_empty[ks]);  // the key slot may be refilled: its mask has been read
            }

            if (t < n_ctx) {
                const int valid = min(BN, ctx - (tb + t) * BN);
                if (valid < BN || bad) {
#pragma unroll
                    for (int i = 0; i < BN; ++i)
                        if (i >= valid || ((bad >> (i >> p.bs_log2)) & 1u)) sv[i] = -INFINITY;
                }
            } else {
                const int lim_t = lim - (t - n_ctx) * BN;
                if (lim_t < BN - 1) {
#pragma unroll
                    for (int i = 0; i < BN; ++i)
                        if (i > lim_t) sv[i] = -INFINITY;
                }
            }
            // row max in the exp2 domain (scale > 0 commutes with max); four independent chains
            // of three-input maxima.  The arithmetic below runs two lanes per instruction
            // where it can: fewer issue slots for the same work leave more to the MMA lanes.
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int e = 0; e < BN / 2; ++e) mx[e & 3] = fmax3(mx[e & 3], sv[2 * e], sv[2 * e + 1]);
            const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.sl2;
            const bool need = mt > m_ref + 8.f;
            float corr = 1.f;
            if (need) {
                corr = ex2(m_ref - mt);
                m_ref = mt;
                l *= corr;
            }
            const float mu = m_ref == -INFINITY ? 0.f : m_ref;
            const float2 sl2v = make_float2(p.sl2, p.sl2), nmu = make_float2(-mu, -mu);
            float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // keys 4k, 4k+1 | 4k+2, 4k+3
            // P in tensor memory is packed here, between the exponentials: the packing is
            // dense integer / FMA work that, as one stretch, would hold the sub-partition's
            // issue slots away from the MMA lanes for hundreds of cycles
            uint32_t ph[BN / 2], pl[BN / 2];  // 16-bit pairs: P (bf16: its hi), and the bf16 lo
#pragma unroll
            for (int e = 0; e < BN / 2; ++e) {
                const float2 x = ffma2(make_float2(sv[2 * e], sv[2 * e + 1]), sl2v, nmu);
                const float a = ex2(x.x), b = ex2(x.y);
                sum2[e & 1] = fadd2(sum2[e & 1], make_float2(a, b));
                if constexpr (C::P_TMEM) {
                    const uint32_t h2 = pack2<BF16>(a, b);
                    ph[e] = h2;
                    if constexpr (BF16) {
                        const float2 d = fsub2(make_float2(a, b),
                                               make_float2(__uint_as_float(h2 << 16), __uint_as_float(h2 & 0xffff0000u)));
                        pl[e] = pack2<BF16>(d.x, d.y);
                    }
                } else {
                    sv[2 * e] = a;
                    sv[2 * e + 1] = b;
                }
            }
            l += (sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y);
            // O must hold every earlier tile before it is rescaled; the P buffer of this tile's
            // parity must have been read by the value MMA of tile t - 2
            if (t > 0 && __any_sync(0xffffffffu, need)) {
                if (!(ok = pfx_warp_wait(&o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, abort_flag, lane))) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < C::DPR / 32; ++c) {
                    float o[32];
                    tmem_ld32(tl + C::COL_O + c * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= corr;
                    tmem_st32(tl + C::COL_O + c * 32, o);
                }
                tmem_wait_st();
            } else if (t > 1) {
                if (!(ok = pfx_warp_wait(&o_done[t & 1], ((t - 2) >> 1) & 1, abort_flag, lane))) break;
            }
            if constexpr (C::P_TMEM) {
                // P row as packed 16-bit pairs into this lane's P columns (bf16: hi, then lo)
                const uint32_t tp = tl + C::COL_P + (t & 1) * C::NP * (BN / 2);
                tmem_st32(tp, *reinterpret_cast<const float(*)[32]>(&ph[0]));
                if constexpr (BF16) tmem_st32(tp + BN / 2, *reinterpret_cast<const float(*)[32]>(&pl[0]));
                tmem_wait_st();
            } else {
                const uint32_t sP = sP0 + (t & 1) * (C::NP * C::P_BYTES);
#pragma unroll
                for (int kc = 0; kc < BN / 8; ++kc) {
                    uint32_t hi[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) hi[e] = pack2<BF16>(sv[kc * 8 + 2 * e], sv[kc * 8 + 2 * e + 1]);
                    sts_v4(sP + kc * (kPfxBM * 16), hi[0], hi[1], hi[2], hi[3]);
                    if constexpr (BF16) {
                        uint32_t lo[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            lo[e] = pack2<BF16>(sv[kc * 8 + 2 * e] - __uint_as_float(hi[e] << 16),
                                                sv[kc * 8 + 2 * e + 1] - __uint_as_float(hi[e] & 0xffff0000u));
                        sts_v4(sP + C::P_BYTES + kc * (kPfxBM * 16), lo[0], lo[1], lo[2], lo[3]);
                    }
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[t & 1]);
        }
        if (ok) ok = pfx_warp_wait(&o_done[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1, abort_flag, lane);
        if (ok && plan.x > 1) {
            // one split of several: O (fp32, relative to the reference max) and the row's
            // (reference max, sum) go to the workspace for the combine
            tc_fence_after();
            const int64_t item = (((int64_t)s * p.Hk + kvh) * p.mt_ws + row0 / kPfxBM) * p.nsplit + split;
            float* wrow = row < rows_total ? p.ws_o + (item * kPfxBM + r) * D : nullptr;
#pragma unroll 1
            for (int c = 0; c < C::DPR / 32; ++c) {
                float o[32];
                tmem_ld32(tl + C::COL_O + c * 32, o);
                tmem_wait_ld();
                if (wrow != nullptr) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (c * 32 + q * 4 < D)
                            *reinterpret_cast<float4*>(wrow + c * 32 + q * 4) =
                                make_float4(o[q * 4], o[q * 4 + 1], o[q * 4 + 2], o[q * 4 + 3]);
                }
            }
            if (wrow != nullptr) p.ws_ml[item * kPfxBM + r] = make_float2(m_ref, l);
        } else if (ok) {
            tc_fence_after();
            const float inv = 1.f / l;
            uint8_t* orow = nullptr;
            if (row < rows_total) {
                const int j = row / G, g = row - j * G;
                orow = static_cast<uint8_t*>(p.out) + ((int64_t)(q0 + j) * p.H + kvh * G + g) * (D * 2);
            }
#pragma unroll 1
            for (int c = 0; c < C::DPR / 32; ++c) {
                float o[32];
                tmem_ld32(tl + C::COL_O + c * 32, o);
                tmem_wait_ld();
                if (orow != nullptr) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int col = c * 32 + q * 8;
                        if (col < D) {
                            uint4 w;
                            w.x = pack2<BF16>(o[q * 8 + 0] * inv, o[q * 8 + 1] * inv);
                            w.y = pack2<BF16>(o[q * 8 + 2] * inv, o[q * 8 + 3] * inv);
                            w.z = pack2<BF16>(o[q * 8 + 4] * inv, o[q * 8 + 5] * inv);
                            w.w = pack2<BF16>(o[q * 8 + 6] * inv, o[q * 8 + 7] * inv);
                            *reinterpret_cast<uint4*>(orow + col * 2) = w;
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kPfxMmaWarp) tmem_dealloc(tm, C::TMEM_COLS);
}

// Merge of a split sequence's partial results, the log-sum-exp combine of softmaxes over
// disjoint key sets: with the splits' reference maxima m_k (exp2 domain), sums l_k and
// un-normalised outputs O_k, out = sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k, M = max m_k.
// One warp per (new token, query head) row; rows of unsplit sequences were written by the
// attention kernel and are skipped.
template <bool BF16>
__global__ void __launch_bounds__(256) pa_prefix_combine_kernel(const PrefixParams p, int D) {
    const int s = blockIdx.y, lane = threadIdx.x & 31;
    const int64_t rr = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);  // j * H + h
    int ctx = p.ctx_lens[s];
    const int q0 = p.qsl[s], q_len = p.qsl[s + 1] - q0;
    if (q_len < 0 || q_len > p.max_query_len || ctx < 0) return;
    ctx = min(ctx, p.mbps * p.bs);
    const int j = (int)(rr / p.H), h = (int)(rr - (int64_t)j * p.H);
    if (j >= q_len) return;
    const int ns = pfx_split_plan((ctx + 63) / 64, p.nsplit, p.split_tiles).x;
    if (ns == 1) return;
    const int kvh = h / p.G, r = j * p.G + (h - kvh * p.G);
    const int64_t item0 = (((int64_t)s * p.Hk + kvh) * p.mt_ws + r / kPfxBM) * p.nsplit;
    const int rt = r % kPfxBM;
    float2 ml = make_float2(-INFINITY, 0.f);
    if (lane < ns) ml = p.ws_ml[(item0 + lane) * kPfxBM + rt];
    float mx = ml.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float w = ml.y > 0.f ? exp2f(ml.x - mx) : 0.f;
    float den = w * ml.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int k = 0; k < ns; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, k);
        const float* orow = p.ws_o + ((item0 + k) * kPfxBM + rt) * D;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int c4 = lane + 32 * i;
            if (c4 < D / 4) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(orow) + c4);
                acc[i].x += wk * v.x;
                acc[i].y += wk * v.y;
                acc[i].z += wk * v.z;
                acc[i].w += wk * v.w;
            }
        }
    }
    const float inv = 1.f / den;
    uint8_t* out = static_cast<uint8_t*>(p.out) + ((int64_t)(q0 + j) * p.H + h) * (D * 2);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int c4 = lane + 32 * i;
        if (c4 < D / 4)
            *reinterpret_cast<uint2*>(out + c4 * 8) =
                make_uint2(pack2<BF16>(acc[i].x * inv, acc[i].y * inv), pack2<BF16>(acc[i].z * inv, acc[i].w * inv));
    }
}

template <bool BF16>
cudaError_t launch_prefix_combine(const PrefixParams& p, int D, dim3 grid, cudaStream_t stream) {
    pa_prefix_combine_kernel<BF16><<<grid, 256, 0, stream>>>(p, D);
    return cudaGetLastError();
}

template <bool BF16, int D>
cudaError_t launch_prefix_kernel(const PrefixParams& p, dim3 grid, cudaStream_t stream) {
    using C = PfxCfg<BF16, D>;
    cudaError_t e = cudaFuncSetAttribute(pa_prefix_kernel<BF16, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    pa_prefix_kernel<BF16, D><<<grid, kPfxThreads, C::SMEM, stream>>>(p);
    return cudaGetLastError();
}

template <bool BF16>
cudaError_t prefix_read_errors(unsigned int* v, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_prefix_errors, sizeof(*v));
    if (e != cudaSuccess || !reset) return e;
    const unsigned int z = 0;
    return cudaMemcpyToSymbol(g_prefix_errors, &z, sizeof(z));
}

}  // namespace pa
