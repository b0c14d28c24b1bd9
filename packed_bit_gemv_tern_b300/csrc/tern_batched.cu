// tern_batched.cu -- one persistent launch for a batch of independent ternary
// products: M = 1 GEMVs, small-M GEMMs and fused SwiGLU pairs (Neutrino-1 8B
// model page: seven coded linears per layer, gate/up feeding a SwiGLU; the
// speculative verifier's M = 7 pass).
//
// Each of the grid's CTAs (one per SM) owns a contiguous run of work units;
// a unit is one 128-row tile (64 gate + 64 up rows for a SwiGLU pair) of one
// item over the item's whole K, so no unit needs a cross-CTA reduction.  The
// host balances the runs by packed bytes.  K is processed in chunks of up to
// 28672 / m codes (the whole K for m = 1 at every Neutrino shape); the B
// operand (activations as two e4m3 terms under a per-row power-of-two scale
// per chunk, see split_pair) and the fp32 accumulators are double buffered
// per chunk, a chunk's B is reused by every later tile of the item on the
// same buffer, and fetching the next chunk's B and reading the previous
// chunk's sums overlap the weight stream.  Roles (17 warps):
//   * warp 0, lane 0: TMA producer; streams every stage of every unit of the
//     CTA through a 6-deep ring of 16 KB stages (128 rows x 512 codes,
//     128-byte swizzle), never waiting on activations.
//   * warps 1-4: bring in B for each chunk (after griddepcontrol.wait), then
//     read the previous chunk's accumulators, rescale and add them into
//     per-row registers, and at the end of a unit write y (scale, SiLU gate).
//     For m = 1 they build B from x themselves; for m >= 2 a short kernel
//     launched just before (k_tern_bprep) has written every chunk's B and row
//     maxima to a workspace once, and a chunk is one bulk copy: building it
//     in every CTA that streams a tile of the item costs more than the
//     chunk's weight stream when m is large.
//   * warps 5-16: three decoder groups of four warps; group g turns the four
//     chunk columns (128 codes of a row each) of the stages s = g (mod 3)
//     into e4m3 +-2/0 bytes (decode8) in TMEM slot g, and lane 0 of warp q
//     of the group then issues the K=32 steps of column q (tcgen05.mma
//     kind::f8f6f4, A from TMEM, B from shared memory, M = 128, N = 16) into
//     the column's accumulator of the chunk's buffer.  Three decoder warps
//     per scheduler hide each other's barrier latency.
// Every mbarrier wait is bounded; on time-out the kernel records the error,
// stops, drains its copies and MMAs, releases its tensor memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "tern.h"
#include "tern_internal.cuh"
#include "tern_mma_common.cuh"
#include "tern_ptx.cuh"

namespace tern {

namespace {

using namespace mma;

constexpr int kMaxItems = 128;             // items per launch (kernel parameter space)
constexpr int kMaxMaps = 144;              // tensor maps per launch: one per item, two per SwiGLU pair
constexpr int kMaxCtas = 160;
constexpr int kThreads = 544;              // 17 warps
constexpr int kFirstStager = 1;            // warps 1-4
constexpr int kStagers = 128;
constexpr int kFirstDec = 5;               // warps 5-16: three decoder groups of four warps
constexpr int kCols = 4;                   // chunk columns of a stage; warp q of a group issues column q
// Decoder group g decodes the stages s = g (mod 3) into TMEM slot g and ring
// slots g and g + 3: every slot a group waits on was last used by the group
// itself, so a phase-parity wait can never be two phases ahead (which would
// alias).
constexpr int kDecGroups = 3;
constexpr int kASlots = 3;                 // TMEM A slots, one stage (128 columns) each
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDCol = kASlots * 128;  // D[buf][k] at kDCol + 16 * (kCols * buf + k)
// B buffer of one chunk in the compact layout: the 2m rows (hi/lo of each
// activation row) of a 16-code block are contiguous, blocks 32m bytes apart.
// The MMA reads eight rows of a core matrix from each block start and eight
// more 128 bytes on, so rows past 2m (ignored D columns) read neighbouring
// blocks' bytes and the last block reads up to 256 bytes past its start.
#ifndef TERN_BBUF_KB
#define TERN_BBUF_KB 56
#endif
constexpr int kBBufBytes = TERN_BBUF_KB * 1024;
constexpr int kBBufStride = kBBufBytes + 256;
// Weight ring depth: 96 KB in flight per SM covers DRAM latency at the HBM
// rate (a plain TMA stream of these stages runs as fast with 6 as with 9);
// the rest of shared memory goes to the two 56 KB activation buffers.  The
// depth is a multiple of kDecGroups (see there).
#ifndef TERN_WSTAGES
#define TERN_WSTAGES 6
#endif
constexpr int kWStages = TERN_WSTAGES;

struct Item {
    const float *scale_g;
    const float *scale_u;
    const uint16_t *x;
    float *y;
    int rows, k, m, swiglu;
    int stages;  // 512-code stages over K
    int cstages; // stages per K chunk (the last may be shorter); a chunk's B fits one buffer
    int unit0;   // first global unit of this item
    int map;     // its codes' tensor map (gate, then up, for a SwiGLU pair)
    // B prepared by k_tern_bprep (nullptr: the staging warps build it): word
    // w of row i of the item's padded K at byte w * 32m + 32i (hi row, then
    // lo row), so chunk c is the contiguous range from c * cstages * 1024m;
    // xmax[8c + i] = the row maximum (fp32 bits of |x|) over chunk c.
    const unsigned char *bsrc;
    const uint32_t *xmax;
};

struct Params {
    int n_items;
    int unit_start[kMaxCtas + 1];  // CTA b runs units [unit_start[b], unit_start[b + 1])
    int item_start[kMaxCtas];      // the item holding unit unit_start[b]
    int stages_cta[kMaxCtas];      // 512-code stages in CTA b's run
    Item item[kMaxItems];
};

struct Maps {
    CUtensorMap m[kMaxMaps];
};

// Shared-memory layout (bytes from the 1024-aligned base).
constexpr uint32_t kOffW = 0;
constexpr uint32_t kOffB = kOffW + kWStages * kStageBytes;
constexpr uint32_t kOffXch = kOffB + 2 * kBBufStride;  // [64][8] fp32
constexpr uint32_t kOffBar = kOffXch + 64 * 8 * 4;
constexpr uint32_t kBarWFull = 0;                       // [kWStages]
constexpr uint32_t kBarWEmpty = kBarWFull + 8 * kWStages;
constexpr uint32_t kBarAEmpty = kBarWEmpty + 8 * kWStages;  // [kASlots]: the slot's MMAs are done
constexpr uint32_t kBarBFull = kBarAEmpty + 8 * kASlots;     // [2]
constexpr uint32_t kBarBEmpty = kBarBFull + 16;
constexpr uint32_t kBarDFull = kBarBEmpty + 16;
constexpr uint32_t kBarDEmpty = kBarDFull + 16;
constexpr uint32_t kBarDrain = kBarDEmpty + 16;  // one commit per issuing warp on exit
constexpr uint32_t kBarTurn = kBarDrain + 8;     // [kCols][kDecGroups]: group g's turn on column q
constexpr uint32_t kWordsOff = kBarTurn + 8 * kCols * kDecGroups;
// words: [0] tmem base, [1] abort, [8..15] xmax buffer 0, [16..23] xmax buffer 1
constexpr uint32_t kSmemBytes = 1024 + kOffBar + kWordsOff + 32 * 4;

__device__ unsigned int g_batched_error;

// Walks the (unit, chunk) sequence of one CTA.  A CTA's units are
// contiguous, so the item index only moves forward; the fields of the current
// item live in registers (a dependent search through the parameter space on
// every unit costs more than a stage of decoding).
struct Cursor {
    const Params *p;
    int unit, unit_end, item, next_unit0, tile, chunk, n_chunks, stages, cstages, n_stages_chunk;
    __device__ void enter_item()
    {
        stages = p->item[item].stages;
        cstages = p->item[item].cstages;
        n_chunks = (stages + cstages - 1) / cstages;
        next_unit0 = item + 1 < p->n_items ? p->item[item + 1].unit0 : 0x7FFFFFFF;
    }
    __device__ void set_chunk() { n_stages_chunk = min(cstages, stages - chunk * cstages); }
    __device__ bool begin(const Params *pp, int b)
    {
        p = pp;
        unit = p->unit_start[b];
        unit_end = p->unit_start[b + 1];
        if (unit >= unit_end) return false;
        item = p->item_start[b];
        enter_item();
        tile = unit - p->item[item].unit0;
        chunk = 0;
        set_chunk();
        return true;
    }
    // Advance one chunk; false at the end of the CTA's run.
    __device__ bool next_chunk()
    {
        if (++chunk < n_chunks) {
            set_chunk();
            return true;
        }
        if (++unit >= unit_end) return false;
        chunk = 0;
        ++tile;
        if (unit >= next_unit0) {  // every item has at least one unit
            ++item;
            enter_item();
            tile = 0;
        }
        set_chunk();
        return true;
    }
    __device__ bool last_chunk_of_unit() const { return chunk + 1 == n_chunks; }
};

// ------------------------------------------------------------------ B prep
// One CTA per (item, chunk, activation row) of the items with m >= 2: the
// row's largest |x| over the chunk, then every word (16 k) of the chunk split
// into its hi and lo e4m3 rows at the row's scale (split_word), written in
// the compact layout the MMA reads (Item::bsrc).  Words past K are zeros.
// The result is the same, byte for byte, as the staging warps' own build.
// A chunk holds at most 28 stages (m = 2), so each thread keeps its words in
// registers between the two passes and all loads are in flight at once.
constexpr int kPrepThreads = 128;
constexpr int kPrepWords = 7;           // words per thread: 28 stages * 32 / 128
constexpr uint32_t kBulkPiece = 16384;  // bytes per bulk copy of a prepared chunk

struct PrepItem {
    const uint16_t *x;
    unsigned char *b;
    uint32_t *xmax;
    int k, m, stages, cstages;
    int task0;  // first task of the item; task task0 + c * m + i is chunk c, row i
};

struct PrepParams {
    int n_items, n_tasks;
    PrepItem item[kMaxItems];
};

__global__ void __launch_bounds__(kPrepThreads) k_tern_bprep(const __grid_constant__ PrepParams p)
{
    __shared__ uint32_t wmax[kPrepThreads / 32];
    // The persistent kernel that follows may start at once: its weight stream
    // needs nothing from here, and its staging warps wait for this grid to
    // finish before they read the workspace.  (A prep CTA fits on an SM
    // beside a persistent CTA.)  The previous kernel on the stream may still
    // read the workspace, and x may come from it: wait for it.
    ptx::grid_dep_launch();
    ptx::grid_dep_wait();
    const int tid = (int)threadIdx.x, task = (int)blockIdx.x;
    int j = 0;
    while (j + 1 < p.n_items && p.item[j + 1].task0 <= task) ++j;
    const PrepItem &it = p.item[j];
    const int local = task - it.task0, c = local / it.m, mm = local - c * it.m;
    const int w0 = c * it.cstages * kStageWords;
    const int nw = min(it.cstages, it.stages - c * it.cstages) * kStageWords;
    const int kw = it.k / 16;
    const uint4 *xr = reinterpret_cast<const uint4 *>(it.x + (size_t)mm * it.k);  // 2 x uint4 per word
    uint4 va[kPrepWords], vb[kPrepWords];
    uint32_t mx = 0;
#pragma unroll
    for (int q = 0; q < kPrepWords; ++q) {
        const int wi = tid + q * kPrepThreads, gw = w0 + wi;
        va[q] = vb[q] = make_uint4(0u, 0u, 0u, 0u);
        if (wi < nw && gw < kw) {
            va[q] = __ldg(xr + 2 * gw);
            vb[q] = __ldg(xr + 2 * gw + 1);
        }
    }
#pragma unroll
    for (int q = 0; q < kPrepWords; ++q) mx = max(mx, max_abs16(va[q], vb[q]));
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if ((tid & 31) == 0) wmax[tid >> 5] = mx;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kPrepThreads / 32; ++w) mx = max(mx, wmax[w]);
    if (tid == 0) it.xmax[8 * c + mm] = mx;
    const float sc = exp2i(row_scale_exp(mx));
    const size_t wbytes = 32u * (size_t)it.m;
    unsigned char *dst = it.b + (size_t)w0 * wbytes + 32u * (size_t)mm;
#pragma unroll
    for (int q = 0; q < kPrepWords; ++q) {
        const int wi = tid + q * kPrepThreads;
        if (wi < nw) {
            uint4 hi4, lo4;
            split_word(va[q], vb[q], sc, hi4, lo4);
            uint4 *d = reinterpret_cast<uint4 *>(dst + (size_t)wi * wbytes);
            d[0] = hi4;
            d[1] = lo4;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
k_tern_batched(const __grid_constant__ Params p, const __grid_constant__ Maps maps)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *gbase = smem_raw + (base - raw);
    const uint32_t wbuf = base + kOffW;
    const uint32_t bbuf = base + kOffB;
    float *xch = reinterpret_cast<float *>(gbase + kOffXch);
    const uint32_t bars = base + kOffBar;
    uint32_t *words = reinterpret_cast<uint32_t *>(gbase + kOffBar + kWordsOff);
    volatile uint32_t *abort_flag = words + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kWStages; ++s) {
            ptx::mbar_init(bars + kBarWFull + 8 * s, 1);
            ptx::mbar_init(bars + kBarWEmpty + 8 * s, 4 * 32);  // every lane of the stage's decoder group
        }
        for (int s = 0; s < kASlots; ++s) ptx::mbar_init(bars + kBarAEmpty + 8 * s, kCols);  // the group's issuing lanes
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bars + kBarBFull + 8 * b, kStagers);  // every staging thread, after its proxy fence
            ptx::mbar_init(bars + kBarBEmpty + 8 * b, kCols);  // the issuing lanes of the chunk's last stage
            ptx::mbar_init(bars + kBarDFull + 8 * b, kCols);
            ptx::mbar_init(bars + kBarDEmpty + 8 * b, 4);
        }
        ptx::mbar_init(bars + kBarDrain, kDecGroups * kCols);
        for (int j = 0; j < kCols * kDecGroups; ++j) ptx::mbar_init(bars + kBarTurn + 8 * j, 1);
        for (int j = 1; j < 32; ++j) words[j] = 0u;
        ptx::fence_proxy_async_smem();
    }
    if (warp == 0) {
        __syncwarp();
        ptx::tmem_alloc(ptx::smem_u32(words), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = words[0];
    if (tid == 0) ptx::grid_dep_launch();
    const Waiter waiter{abort_flag, &g_batched_error};
    Cursor cur;
    const bool any = cur.begin(&p, (int)blockIdx.x);

    if (warp == 0) {
        // --------------------------------------------------------- producer
        // "Empty" barriers are waited at the flipped parity: a fresh barrier
        // counts its preceding phase as complete, so the first pass through
        // the ring needs no special case.
        if (lane == 0 && any) {
            int gs = 0, slot = 0;
            uint32_t par = 0;
            bool more = true;
            while (more) {
                const Item &it = p.item[cur.item];
                const int row0 = cur.tile * (it.swiglu ? 64 : 128);
                for (int st = 0; st < cur.n_stages_chunk; ++st, ++gs) {
                    const uint32_t empty = bars + kBarWEmpty + 8 * slot;
                    if (!ptx::mbar_try_wait(empty, par ^ 1u) && !waiter.wait(empty, par ^ 1u)) {
                        more = false;
                        break;
                    }
                    const uint32_t dst = wbuf + slot * kStageBytes, full = bars + kBarWFull + 8 * slot;
                    const int c0 = (cur.chunk * cur.cstages + st) * kStageWords;
                    ptx::mbar_arrive_expect_tx(full, kStageBytes);
                    ptx::tma_load_2d(dst, &maps.m[it.map], c0, row0, full);
                    if (it.swiglu) ptx::tma_load_2d(dst + kStageBytes / 2, &maps.m[it.map + 1], c0, row0, full);
                    if (++slot == kWStages) {
                        slot = 0;
                        par ^= 1u;
                    }
                }
                more = more && cur.next_chunk();
            }
            for (int s = gs > kWStages ? gs - kWStages : 0; s < gs; ++s)
                drain_wait(bars + kBarWFull + 8 * (s % kWStages), (s / kWStages) & 1, &g_batched_error);
        }
    } else if (warp >= kFirstDec) {
        // ----------------------------------------- decoders and MMA issuers
        // Group g decodes all four columns of the stages s = g (mod 3) into
        // TMEM slot g (quad q owns TMEM lanes 32q..32q+31), the group meets
        // at a named barrier, and then warp q issues the four K=32 steps of
        // column q (tcgen05.mma kind::f8f6f4, A from TMEM, B from shared
        // memory, M = 128, N = 16) into D[buf][q].  Stage s's MMAs on a column
        // follow stage s-1's, issued by the previous group, through that
        // column's turn barriers (tcgen05 fence, mbarrier, fence), which order
        // the accumulation; a warp issues for one stage in three, so one
        // thread's waits and bookkeeping overlap the others' MMA issue (a
        // warp issues an MMA about every 54 cycles, warps overlap).  Every
        // slot a group waits on was last used by the group itself, so no
        // phase-parity wait runs two phases ahead of its barrier.  A chunk's
        // first-stage issuers wait for its B and D buffers (later stages see
        // them through the turn chain); its last-stage issuers commit the
        // chunk's D and B, which tracks the whole accumulation chain.
        const int g = (warp - kFirstDec) >> 2;
        const int quad = warp & 3;
        const int i = quad * 32 + lane;
        const uint32_t tm_row = tmem + ((uint32_t)(quad * 32) << 16);
        const uint32_t row_addr = wbuf + (uint32_t)i * 128u;
        const uint32_t sw = (uint32_t)(i & 7);  // 128-byte swizzle: 16-byte chunk c of row i sits at c ^ (i & 7)
        const uint32_t a_col = tmem + (uint32_t)(g * 128 + quad * 32);  // column q of slot g (lane 0)
        const uint32_t my_turn = bars + kBarTurn + 8u * (uint32_t)(kDecGroups * quad + g);
        const uint32_t next_turn = bars + kBarTurn + 8u * (uint32_t)(kDecGroups * quad + (g + 1) % kDecGroups);
        const uint32_t a_empty = bars + kBarAEmpty + 8u * (uint32_t)g;
        const uint32_t bar_id = 2u + (uint32_t)g;  // 0: __syncthreads, 1: staging warps
        static_assert(kWStages % kDecGroups == 0 && kASlots == kDecGroups, "slots must cycle within a group");
        int w_r = g, w_q = 0;      // stage s: ring slot s % kWStages, use s / kWStages
        int a_q = 0;               //          TMEM slot g, use s / kASlots
        uint32_t tpar = g == 0 ? 1u : 0u;  // stage 0 needs no turn
        int gs = 0, gc = 0;
        bool more = any;
        while (more) {
            const int n_st = cur.n_stages_chunk;
            const int buf = gc & 1;
            const uint32_t wbytes = 32u * (uint32_t)p.item[cur.item].m;
            for (int st = (g - gs % kDecGroups + kDecGroups) % kDecGroups; st < n_st; st += kDecGroups) {
                const uint32_t wf = bars + kBarWFull + 8 * w_r;
                const uint32_t wpar = (uint32_t)w_q & 1u, apar = (uint32_t)a_q & 1u;
                // both fast-path tests issue back to back; the bounded waits only on a miss
                bool okw = ptx::mbar_try_wait(wf, wpar);
                bool oka = ptx::mbar_try_wait(a_empty, apar ^ 1u);
                if (!okw) okw = waiter.wait(wf, wpar);
                if (okw && !oka) oka = waiter.wait(a_empty, apar ^ 1u);
                if (__all_sync(0xFFFFFFFFu, okw && oka)) {
                    ptx::tc_fence_after();
                    const uint32_t srow = row_addr + (uint32_t)w_r * kStageBytes;
                    const uint32_t ta = tm_row + (uint32_t)(g * 128);
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        const uint4 v0 = ptx::lds128(srow + ((((uint32_t)(2 * c)) ^ sw) << 4));
                        const uint4 v1 = ptx::lds128(srow + ((((uint32_t)(2 * c + 1)) ^ sw) << 4));
                        uint32_t r[32];
                        decode8(v0, v1, r);
                        ptx::tmem_st_32x32b_x32(ta + 32u * (uint32_t)c, r);
                    }
                    ptx::mbar_arrive(bars + kBarWEmpty + 8 * w_r);  // after the last store, which consumed the loads
                    ptx::tmem_wait_st();
                }
                ptx::tc_fence_before();
                // the group's 128 rows are in TMEM; stop together on an abort
                if (ptx::named_bar_or(bar_id, 128, *abort_flag != 0u)) {
                    more = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t bpar = (uint32_t)(gc >> 1) & 1u;
                    const uint32_t bfull = bars + kBarBFull + 8 * buf, dempty = bars + kBarDEmpty + 8 * buf;
                    bool lok = st != 0 || ((ptx::mbar_try_wait(bfull, bpar) || waiter.wait(bfull, bpar)) &&
                                           (ptx::mbar_try_wait(dempty, bpar ^ 1u) || waiter.wait(dempty, bpar ^ 1u)));
                    lok = lok && (ptx::mbar_try_wait(my_turn, tpar) || waiter.wait(my_turn, tpar));
                    if (lok) {
                        ptx::tc_fence_after();
                        const uint32_t d = tmem + kDCol + 16u * (uint32_t)(kCols * buf + quad);
                        // compact B: 16-code blocks 32m bytes apart; column q of stage st at word st*32 + 8q
                        const uint64_t bd = b_desc_lbo(bbuf + (uint32_t)buf * kBBufStride +
                                                           (uint32_t)(st * kStageWords + 8 * quad) * wbytes,
                                                       wbytes);
                        const uint32_t bd_lo = (uint32_t)bd, bd_hi = (uint32_t)(bd >> 32), t_step = (2u * wbytes) >> 4;
                        ptx::mma_ts_f8f6f4_lh(d, a_col, bd_lo, bd_hi, kIdesc, st != 0 ? 1u : 0u);
#pragma unroll
                        for (int t = 1; t < 4; ++t)  // K=32 step 4q+t: A columns +8t, B words +2t
                            ptx::mma_ts_f8f6f4_lh(d, a_col + 8u * t, bd_lo + t_step * t, bd_hi, kIdesc, 1u);
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(next_turn);  // the next stage's MMAs on this column follow these
                        ptx::mma_commit(a_empty);
                        if (st == n_st - 1) {
                            ptx::mma_commit(bars + kBarDFull + 8 * buf);
                            ptx::mma_commit(bars + kBarBEmpty + 8 * buf);
                        }
                    }
                }
                __syncwarp();
                tpar ^= 1u;
                w_r += kDecGroups;  // s += 3
                if (w_r >= kWStages) {
                    w_r -= kWStages;
                    ++w_q;
                }
                ++a_q;
            }
            gs += n_st;
            ++gc;
            more = more && cur.next_chunk();
        }
        // arrives once every MMA this thread issued has completed (at once if none)
        if (lane == 0) ptx::mma_commit(bars + kBarDrain);
    } else {
        // ------------------------------------------- B staging and epilogue
        const int st_tid = tid - 32 * kFirstStager;  // 0..127
        const int quad = warp & 3;
        const int i = quad * 32 + lane;               // tile row == TMEM lane
        ptx::grid_dep_wait();
        float acc[8];
#pragma unroll
        for (int n = 0; n < 8; ++n) acc[n] = 0.f;
        // previous chunk, whose accumulators are read after the next chunk's B is staged
        int prev_item = -1, prev_tile = 0;
        bool prev_last = false;
        int gc = 0;
        bool ok = any;
        // what each B buffer holds: a chunk of an item is staged once and reused
        // by every later tile of the same item that lands on this buffer
        int held_item[2] = {-1, -1}, held_chunk[2] = {-1, -1};
        int last_gc[2] = {-1, -1};  // last chunk whose BFull phase each buffer took part in

        auto epilogue = [&](int e) {  // read chunk e's accumulators, finish the unit if it was its last chunk
            const int eb = e & 1;
            uint32_t good = 1u;
            if (lane == 0) good = waiter.wait(bars + kBarDFull + 8 * eb, (e >> 1) & 1) ? 1u : 0u;
            good = __shfl_sync(0xFFFFFFFFu, good, 0);
            float dsum[16];
#pragma unroll
            for (int n = 0; n < 16; ++n) dsum[n] = 0.f;
            if (good) {
                ptx::tc_fence_after();
#pragma unroll 1
                for (int a = 0; a < kCols; ++a) {
                    uint32_t dv[16];
                    ptx::tmem_ld_32x32b_x16(tmem + ((uint32_t)(quad * 32) << 16) + kDCol + 16u * (kCols * eb + a), dv);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int n = 0; n < 16; ++n) dsum[n] += __uint_as_float(dv[n]);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bars + kBarDEmpty + 8 * eb);
            const Item &it = p.item[prev_item];
            const uint32_t *xm = words + 8 + 8 * eb;
#pragma unroll
            for (int mm = 0; mm < 8; ++mm) {
                if (mm < it.m) {
                    const int s = row_scale_exp(xm[mm]);
                    acc[mm] += dsum[2 * mm] * exp2i(-s) + dsum[2 * mm + 1] * exp2i(max(-s - 4, -126));
                }
            }
            if (!prev_last) return;
            if (it.swiglu) {
                const int r = prev_tile * 64 + (i & 63);
                if (i >= 64 && r < it.rows) {
                    const float su = it.scale_u[r];
#pragma unroll
                    for (int n = 0; n < 8; ++n) xch[(i - 64) * 8 + n] = su * (0.5f * acc[n]);
                }
                ptx::named_bar_sync(1, kStagers);
                if (i < 64 && r < it.rows) {
                    const float sg = it.scale_g[r];
#pragma unroll
                    for (int n = 0; n < 8; ++n)
                        if (n < it.m) it.y[(size_t)n * it.rows + r] = silu_f(sg * (0.5f * acc[n])) * xch[i * 8 + n];
                }
                ptx::named_bar_sync(1, kStagers);  // xch reusable
            } else {
                const int r = prev_tile * 128 + i;
                if (r < it.rows) {
                    const float sc = it.scale_g[r];
#pragma unroll
                    for (int n = 0; n < 8; ++n)
                        if (n < it.m) it.y[(size_t)n * it.rows + r] = sc * (0.5f * acc[n]);
                }
            }
#pragma unroll
            for (int n = 0; n < 8; ++n) acc[n] = 0.f;
        };

        while (ok) {
            const int buf = gc & 1;
            const Item &it = p.item[cur.item];
            // the MMAs of chunk gc-2 must be done with this B buffer
            if (lane == 0) waiter.wait(bars + kBarBEmpty + 8 * buf, ((gc >> 1) & 1) ^ 1);
            uint32_t *xm = words + 8 + 8 * buf;
            const bool reuse = held_item[buf] == cur.item && held_chunk[buf] == cur.chunk;
            // Past this barrier every staging warp has finished chunk gc-2's
            // epilogue, the last reader of this buffer's row maxima xm.  The
            // barrier ORs the abort flag over the four staging warps, so they
            // all take the same branch.
            if (ptx::named_bar_or(1, kStagers, *abort_flag != 0u)) break;
            if (reuse) {  // B (and its row scales) already hold this chunk
                last_gc[buf] = gc;
                ptx::mbar_arrive(bars + kBarBFull + 8 * buf);
                if (gc >= 1) epilogue(gc - 1);
                prev_item = cur.item;
                prev_tile = cur.tile;
                prev_last = cur.last_chunk_of_unit();
                ++gc;
                ok = cur.next_chunk();
                continue;
            }
            const int n_words = cur.n_stages_chunk * kStageWords;
            const int k0 = cur.chunk * cur.cstages * kStageWords * 16;
            const int m = it.m;
            const int n_items = m * n_words;
            const uint32_t bb = bbuf + (uint32_t)buf * kBBufStride;
            const uint32_t wbytes = 32u * (uint32_t)m;  // compact B: a block holds rows 0..2m-1
            const uint32_t bfull = bars + kBarBFull + 8 * buf;
            if (it.bsrc != nullptr) {
                // prepared: the chunk's bytes in a few bulk copies that
                // complete on BFull (its phase also waits for every staging
                // thread's arrival below), and the chunk's row maxima
                if (st_tid == 0) {
                    const uint32_t bytes = (uint32_t)n_words * wbytes;
                    const unsigned char *src = it.bsrc + (size_t)(k0 / 16) * wbytes;
                    ptx::mbar_expect_tx(bfull, bytes);
                    for (uint32_t o = 0; o < bytes; o += kBulkPiece)
                        ptx::bulk_load(bb + o, src + o, min(kBulkPiece, bytes - o), bfull);
                }
                if (st_tid < m) xm[st_tid] = it.xmax[8 * cur.chunk + st_tid];
                held_item[buf] = cur.item;
                held_chunk[buf] = cur.chunk;
                last_gc[buf] = gc;
                ptx::mbar_arrive(bfull);
                if (gc >= 1) epilogue(gc - 1);
                prev_item = cur.item;
                prev_tile = cur.tile;
                prev_last = cur.last_chunk_of_unit();
                ++gc;
                ok = cur.next_chunk();
                continue;
            }
            if (st_tid < 8) xm[st_tid] = 0u;
            ptx::named_bar_sync(1, kStagers);
            // The compact layout keeps 32 bytes (hi and lo rows) per 16
            // activations of a row, the size of the 16 bf16 values, so each
            // word is copied asynchronously to its final place (all copies in
            // flight at once, zero-filled past K), its row maximum reduced
            // from shared memory, and split in place.  A warp's 32 items are
            // 32 consecutive words of one activation row (n_words is a
            // multiple of 32), so the maximum is reduced in the warp first.
            for (int item = st_tid; item < n_items; item += kStagers) {
                const int mm = item / n_words, wi = item - mm * n_words;
                const int kk = k0 + 16 * wi;
                const bool in_k = kk < it.k;
                const uint16_t *src = in_k ? it.x + (size_t)mm * it.k + kk : it.x;
                const uint32_t at = bb + (uint32_t)wi * wbytes + 32u * (uint32_t)mm;
                ptx::cp_async16(at, src, in_k ? 16u : 0u);
                ptx::cp_async16(at + 16u, src + 8, in_k ? 16u : 0u);
            }
            ptx::cp_async_wait_all();
            for (int item = st_tid; item < n_items; item += kStagers) {
                const int mm = item / n_words, wi = item - mm * n_words;
                const uint32_t at = bb + (uint32_t)wi * wbytes + 32u * (uint32_t)mm;
                const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, max_abs16(ptx::lds128(at), ptx::lds128(at + 16u)));
                if (lane == 0) atomicMax(&xm[mm], mx);
            }
            ptx::named_bar_sync(1, kStagers);
            for (int item = st_tid; item < n_items; item += kStagers) {
                const int mm = item / n_words, wi = item - mm * n_words;
                const uint32_t at = bb + (uint32_t)wi * wbytes + 32u * (uint32_t)mm;
                uint4 hi4, lo4;
                split_word(ptx::lds128(at), ptx::lds128(at + 16u), exp2i(row_scale_exp(xm[mm])), hi4, lo4);
                ptx::sts128(at, hi4);
                ptx::sts128(at + 16u, lo4);
            }
            held_item[buf] = cur.item;
            held_chunk[buf] = cur.chunk;
            last_gc[buf] = gc;
            ptx::fence_proxy_async_smem();  // my B writes -> visible to the tensor core
            ptx::mbar_arrive(bfull);
            if (gc >= 1) epilogue(gc - 1);
            prev_item = cur.item;
            prev_tile = cur.tile;
            prev_last = cur.last_chunk_of_unit();
            ++gc;
            ok = cur.next_chunk();
        }
        if (!ptx::named_bar_or(1, kStagers, *abort_flag != 0u) && gc >= 1) epilogue(gc - 1);
        // After an abort a bulk copy into a B buffer may still be in flight:
        // its buffer's last BFull phase completes only when it has landed
        // (every staging thread has arrived on it).
        if (st_tid == 0)
            for (int b = 0; b < 2; ++b)
                if (last_gc[b] >= 0)
                    drain_wait(bars + kBarBFull + 8 * b, (uint32_t)(last_gc[b] >> 1) & 1u, &g_batched_error);
    }

    __syncthreads();
    if (warp == 0) {
        // every MMA of this CTA has completed before its tensor memory is released
        if (lane == 0) drain_wait(bars + kBarDrain, 0, &g_batched_error);
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// Launch groups of a batch: consecutive runs of items, each with up to
// kMaxItems items that have rows > 0 and k > 0 ("real" items) holding up to
// kMaxMaps tensor maps.  The fewest groups a greedy walk needs is found
// first, then the real items are spread evenly over that many groups (a
// short last launch streams far below the rate of a full one).  Items with
// rows == 0 (nothing to do) or k == 0 (y = 0, written by a small CUDA-core
// launch of their own) ride along without counting.  Returns the end index of
// each group.
std::vector<int> plan_groups(const tern_batch_item *items, int n)
{
    auto walk = [&](int per_group) {
        std::vector<int> ends;
        int cnt = 0, n_maps = 0;
        for (int idx = 0; idx < n; ++idx) {
            const tern_batch_item &b = items[idx];
            if (b.w->rows == 0 || b.w->k == 0) continue;
            const int need = b.up ? 2 : 1;
            if (cnt == per_group || n_maps + need > kMaxMaps) {
                ends.push_back(idx);
                cnt = 0;
                n_maps = 0;
            }
            ++cnt;
            n_maps += need;
        }
        ends.push_back(n);
        return ends;
    };
    int real = 0;
    for (int idx = 0; idx < n; ++idx) real += (items[idx].w->rows != 0 && items[idx].w->k != 0) ? 1 : 0;
    const std::vector<int> greedy = walk(kMaxItems);
    if (greedy.size() <= 1) return greedy;
    const int per = (real + (int)greedy.size() - 1) / (int)greedy.size();
    std::vector<int> even = walk(per);
    return even.size() <= greedy.size() ? even : greedy;
}

// Workspace of prepared activations per (device, stream), grown on demand.
// A grown-out buffer is never freed: a launch captured in a CUDA graph keeps
// the address it was captured with.  Returns nullptr if the allocation fails
// (the staging warps then build B themselves).
void *workspace(cudaStream_t stream, size_t need)
{
    struct Buf {
        void *p = nullptr;
        size_t bytes = 0;
    };
    static std::mutex mu;
    static std::map<std::pair<int, cudaStream_t>, Buf> all;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    Buf &b = all[{dev, stream}];
    if (b.bytes >= need) return b.p;
    const size_t bytes = need > 2 * b.bytes ? need : 2 * b.bytes;
    // an allocation is allowed while a stream of this thread is being captured
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    if (cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess) return nullptr;
    void *p = nullptr;
    const cudaError_t e = cudaMalloc(&p, bytes);
    cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    b.p = p;
    b.bytes = bytes;
    return p;
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// 512-code stages over K, and stages per chunk: the fewest chunks that fit a
// B buffer, of equal stage counts (a short last chunk would pay the
// per-chunk costs for little work).
void chunk_plan(int k, int m, int &stages, int &cstages)
{
    stages = (k / 16 + kStageWords - 1) / kStageWords;
    const int cap = kBBufBytes / (1024 * m);  // stages of compact B one buffer holds
    const int n_chunks = (stages + cap - 1) / cap;
    cstages = (stages + n_chunks - 1) / n_chunks;
}

// Workspace bytes of one prepared item (see Item::bsrc, Item::xmax).
size_t prep_bytes(int stages, int cstages, int m)
{
    const int n_chunks = (stages + cstages - 1) / cstages;
    return align256((size_t)stages * 1024u * (size_t)m) + align256((size_t)n_chunks * 8u * sizeof(uint32_t));
}

// Scratch of tern_gemm_batched_noalloc: module-scope device memory, which the
// CUDA runtime sets up when it loads the library's kernels on a device, so
// the entry point itself never allocates.
__device__ __align__(256) unsigned char g_noalloc_ws[TERN_NOALLOC_WS_BYTES];

}  // namespace

int batched_launches(const tern_batch_item *items, int n)
{
    int launches = 0, begin = 0;
    for (const int end : plan_groups(items, n)) {
        bool any = false, prep = false;
        for (int i = begin; i < end; ++i) {
            if (items[i].w->rows == 0) continue;
            if (items[i].w->k == 0) {
                ++launches;
            } else {
                any = true;
                prep = prep || items[i].m >= 2;
            }
        }
        launches += (any ? 1 : 0) + (prep ? 1 : 0);
        begin = end;
    }
    return launches;
}

namespace {

// Launches the batch.  fixed_ws: a workspace the caller guarantees to be
// large enough for every launch group (nullptr: the per-stream workspace).
tern_status run_batched(const tern_batch_item *items, int n, cudaStream_t stream, unsigned char *fixed_ws)
{
    static_assert(sizeof(Params) + sizeof(Maps) < 32000, "kernel parameters exceed 32 KB");
    const int sms = sm_count();
    // the kernel's shared-memory attribute, once per device
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TERN_ERR_CUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(k_tern_batched, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
            cudaSuccess)
            return TERN_ERR_CUDA;
        attr_set[dev] = true;
    }
    int begin = 0;
    for (const int end : plan_groups(items, n)) {
        Params prm;
        std::memset(&prm, 0, sizeof(prm));
        Maps maps;
        std::memset(&maps, 0, sizeof(maps));
        std::vector<long long> unit_cost;
        int cnt = 0, units = 0, n_maps = 0;
        for (int idx = begin; idx < end; ++idx) {
            const tern_batch_item &b = items[idx];
            if (b.w->rows == 0) continue;
            if (b.w->k == 0) {  // empty sum: y = scale * 0
                const tern_status st = gemm_cc(b.w, b.up, b.x, b.m, b.y, stream);
                if (st != TERN_OK) return st;
                continue;
            }
            Item &it = prm.item[cnt];
            it.scale_g = b.w->scale;
            it.scale_u = b.up ? b.up->scale : nullptr;
            it.x = b.x;
            it.y = b.y;
            it.rows = b.w->rows;
            it.k = b.w->k;
            it.m = b.m;
            it.swiglu = b.up != nullptr;
            chunk_plan(it.k, it.m, it.stages, it.cstages);
            it.unit0 = units;
            it.map = n_maps;
            const int tile_rows = it.swiglu ? 64 : 128;
            const int tiles = (it.rows + tile_rows - 1) / tile_rows;
            if (!make_code_map(&maps.m[n_maps++], b.w->codes, it.rows, it.k / 16, tile_rows)) return TERN_ERR_CUDA;
            if (it.swiglu && !make_code_map(&maps.m[n_maps++], b.up->codes, it.rows, it.k / 16, tile_rows))
                return TERN_ERR_CUDA;
            for (int t = 0; t < tiles; ++t) unit_cost.push_back(it.stages);
            units += tiles;
            ++cnt;
        }
        begin = end;
        if (cnt == 0) continue;
        prm.n_items = cnt;

        // Items with m >= 2 take their B from the workspace, written by one
        // k_tern_bprep launch just before: per item the padded K's words
        // (1024m bytes per stage), then 8 row maxima per chunk.
        PrepParams pp;
        std::memset(&pp, 0, sizeof(pp));
        size_t ws_need = 0;
        std::vector<std::pair<size_t, size_t>> ws_off(cnt);
        for (int j = 0; j < cnt; ++j) {
            const Item &it = prm.item[j];
            if (it.m < 2) continue;
            const int n_chunks = (it.stages + it.cstages - 1) / it.cstages;
            if (it.cstages * kStageWords > kPrepWords * kPrepThreads) return TERN_ERR_SHAPE;  // cannot happen: m >= 2
            ws_off[j].first = ws_need;
            ws_off[j].second = ws_need + align256((size_t)it.stages * 1024u * (size_t)it.m);
            ws_need += prep_bytes(it.stages, it.cstages, it.m);
        }
        unsigned char *ws = nullptr;
        if (ws_need > 0) ws = fixed_ws != nullptr ? fixed_ws : static_cast<unsigned char *>(workspace(stream, ws_need));
        if (ws != nullptr) {
            for (int j = 0; j < cnt; ++j) {
                Item &it = prm.item[j];
                if (it.m < 2) continue;
                it.bsrc = ws + ws_off[j].first;
                it.xmax = reinterpret_cast<const uint32_t *>(ws + ws_off[j].second);
                PrepItem &q = pp.item[pp.n_items++];
                q.x = it.x;
                q.b = ws + ws_off[j].first;
                q.xmax = reinterpret_cast<uint32_t *>(ws + ws_off[j].second);
                q.k = it.k;
                q.m = it.m;
                q.stages = it.stages;
                q.cstages = it.cstages;
                q.task0 = pp.n_tasks;
                pp.n_tasks += (it.stages + it.cstages - 1) / it.cstages * it.m;
            }
            cudaLaunchConfig_t pcfg = {};
            pcfg.gridDim = dim3((unsigned)pp.n_tasks, 1, 1);
            pcfg.blockDim = dim3(kPrepThreads, 1, 1);
            pcfg.stream = stream;
            cudaLaunchAttribute pattr;
            pattr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
            pattr.val.programmaticStreamSerializationAllowed = 1;
            pcfg.attrs = &pattr;
            pcfg.numAttrs = 1;
            if (cudaLaunchKernelEx(&pcfg, k_tern_bprep, pp) != cudaSuccess) return TERN_ERR_CUDA;
        }
        // contiguous runs of units with balanced stage counts
        const int ctas = units < sms ? units : (sms < kMaxCtas ? sms : kMaxCtas);
        long long total = 0;
        for (long long c : unit_cost) total += c;
        int u = 0;
        long long acc = 0;
        prm.unit_start[0] = 0;
        for (int b = 1; b < ctas; ++b) {
            const long long target = total * b / ctas;
            while (u < units && acc + unit_cost[u] / 2 < target) acc += unit_cost[u++];
            prm.unit_start[b] = u;
        }
        prm.unit_start[ctas] = units;
        for (int b = 0, j = 0; b < ctas; ++b) {
            while (j + 1 < cnt && prm.item[j + 1].unit0 <= prm.unit_start[b]) ++j;
            prm.item_start[b] = j;
        }
        for (int b = 0; b < ctas; ++b) {
            long long st = 0;
            for (int q = prm.unit_start[b]; q < prm.unit_start[b + 1]; ++q) st += unit_cost[q];
            prm.stages_cta[b] = (int)st;
        }

        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)ctas, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, k_tern_batched, prm, maps) != cudaSuccess) return TERN_ERR_CUDA;
        if (cudaGetLastError() != cudaSuccess) return TERN_ERR_CUDA;
    }
    return TERN_OK;
}

}  // namespace

tern_status gemm_batched(const tern_batch_item *items, int n, cudaStream_t stream)
{
    return run_batched(items, n, stream, nullptr);
}

tern_status gemm_batched_noalloc(const tern_batch_item *items, int n, cudaStream_t stream)
{
    // every launch group's prepared activations must fit the static scratch
    // (the groups run one after another on the stream and reuse it)
    int begin = 0;
    for (const int end : plan_groups(items, n)) {
        size_t need = 0;
        for (int i = begin; i < end; ++i) {
            const tern_batch_item &b = items[i];
            if (b.w->rows == 0 || b.w->k == 0 || b.m < 2) continue;
            int stages = 0, cstages = 0;
            chunk_plan(b.w->k, b.m, stages, cstages);
            need += prep_bytes(stages, cstages, b.m);
        }
        if (need > (size_t)TERN_NOALLOC_WS_BYTES) return TERN_ERR_SHAPE;
        begin = end;
    }
    // the scratch's device address, looked up once per device
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TERN_ERR_CUDA;
    void *ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (addr[dev] == nullptr && cudaGetSymbolAddress(&addr[dev], g_noalloc_ws) != cudaSuccess) {
            addr[dev] = nullptr;
            return TERN_ERR_CUDA;
        }
        ws = addr[dev];
    }
    return run_batched(items, n, stream, static_cast<unsigned char *>(ws));
}

tern_status take_batched_error()
{
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_batched_error, sizeof(v)) != cudaSuccess) return TERN_ERR_CUDA;
    if (v != 0u) {
        if (cudaMemcpyToSymbol(g_batched_error, &z, sizeof(z)) != cudaSuccess) return TERN_ERR_CUDA;
        return TERN_ERR_TIMEOUT;
    }
    return TERN_OK;
}

}  // namespace tern
