// tern_mma.cu -- tensor-core ternary GEMV / small-M GEMM for sm_103a.
//
// What is computed (Neutrino-1 8B model page, intro: the ternary weights stay
// bit-packed and are decoded inside the matrix kernels; spec table: gated
// SwiGLU feed-forward; "Where the bytes live": per-row scales):
//     y[m][r] = scale[r] * sum_k t[r][k] x[m][k]      m < M (M <= 8)
//     h[m][r] = silu(y_gate[m][r]) * y_up[m][r]       (SwiGLU pair)
//
// Layout of the work: one CTA per SM owns 128 weight rows (the MMA's M) and
// one K range; a cluster of S CTAs splits K and reduces through distributed
// shared memory.  Roles (13 warps):
//   * warp 0, lane 0: TMA producer.  2-D tiled bulk copies bring 128 rows x
//     512 codes (16 KB, 128-byte swizzle) per stage into a shared-memory ring.
//     Weights do not depend on the previous kernel, so the first stages are
//     requested before anything waits on it (programmatic dependent launch).
//   * warps 1-4: B operand staging.  After griddepcontrol.wait they turn the
//     activations of the K range into the MMA's B operand.  Each bf16 value x
//     of activation row i goes to one of two magnitude bands.  Band A holds
//     the elements with |x| >= 2^(e-13), where 2^e <= max|x| < 2^(e+1) over
//     the row; band B the others, with 2^f <= max over band B < 2^(f+1).  In
//     its band, x is split into two e4m3 terms under the band's power-of-two
//     scale 2^s (the band maximum lands in [128, 256)):
//     x*2^s = hi + lo/16, hi = RN_e4m3(x*2^s), lo = RN_e4m3((x*2^s - hi)*16).
//     A bf16 value has 8 significant bits and each e4m3 term holds 4, so a
//     band's split is exact for every element at least 2^-13 of its band
//     maximum: band A always, band B for |x| >= 2^(f-13); smaller elements
//     carry an absolute error of at most 2^(f-21).  B rows 4i .. 4i+3 hold
//     hi_A, lo_A, hi_B, lo_B of row i (N = 16 for m <= 4, 32 above).
//   * warps 5-12: two decoder warpgroups taking alternate chunks of 8 words
//     (128 codes) per row.  Thread i owns weight row i (TMEM lane i).  Each
//     32-bit word (16 codes) becomes four registers of four e4m3 bytes:
//         R_j = (w << (6 - 2j)) & 0xC0C0C0C0,   byte b of R_j <- code 4b + j
//     which puts b1 on the sign bit and b0 on the exponent's top bit: exactly
//     0, +2 or -2 in e4m3 (the invalid code 10 gives -0).  No multiply touches
//     a weight.  The 32 registers go to the chunk's TMEM slot (tcgen05.st);
//     the group's four warps meet at a named barrier, then warp q issues the
//     chunk's K=32 step q (tcgen05.mma kind::f8f6f4, A e4m3 from TMEM, B e4m3
//     from shared memory, M = 128, N = 16 or 32) into its own fp32
//     accumulator D[q] and commits the slot back.  Spreading the issue over eight warps
//     keeps the per-thread issue cost (about 45 cycles per MMA) off the
//     critical path.
//   * epilogue: the four accumulators are summed (tcgen05.ld), the hi/lo
//     columns of each band rescaled by 2^-s and 2^-(s+4), split-K partials
//     pushed into rank 0's
//     shared memory and summed there in rank order after one cluster barrier,
//     then y = scale * (0.5 * sum) (the weights entered as +-2), or
//     silu(gate) * up for the SwiGLU pair (tile rows 0-63 are gate rows,
//     64-127 the matching up rows).
// Every mbarrier wait is bounded; on time-out the kernel records the error,
// stops, waits for its own copies and MMAs, releases its tensor memory and
// returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>
#include <unordered_map>

#include "tern.h"
#include "tern_internal.cuh"
#include "tern_mma_common.cuh"
#include "tern_ptx.cuh"

namespace tern {

namespace {

constexpr int kThreads = 416;             // 13 warps
constexpr int kStagerWarps = 4;           // warps 1-4: B operand staging, then MMA issue
constexpr int kStagers = 32 * kStagerWarps;
constexpr int kIssuers = kStagerWarps;    // one MMA issuer (lane 0) per staging warp
constexpr int kFirstDecWarp = 1 + kStagerWarps;  // warps 5-12: decoders (two warpgroups)
constexpr int kChunkWords = 8;            // words per row per decode chunk (2 x 16 B)
constexpr int kASlots = 3;                // TMEM A slots, one stage (128 columns) each
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDCol = kASlots * 128;  // accumulators D[k], k < kIssuers, at kDCol + N k
constexpr int kMaxWStages = 8;
// Every CTA allocates all 512 TMEM columns.  Asking for more than half of the
// SM's shared memory keeps one CTA per SM, so tcgen05.alloc never waits for a
// CTA of the same launch (which could itself be waiting, at a cluster barrier,
// on the one that waits).
constexpr uint32_t kMinSmem = 118 * 1024;

__device__ unsigned int g_mma_error;  // bit 0: a bounded wait ran out

struct MmaParams {
    const float *scale_g;
    const float *scale_u;
    const uint16_t *x;
    float *y;
    int rows;
    int k;
    int m;            // activation rows (1..8)
    int total_st;     // stages over the whole K
    int per_st;       // stages per cluster rank
    int split;        // cluster size
    int n_wst;        // shared-memory weight ring depth
    long long wait_limit;  // bound of every Waiter, in cycles
    uint32_t off_b;   // shared-memory byte offsets from the 1024-aligned base
    uint32_t off_red;
    uint32_t off_xch;
    uint32_t off_bar;
};

// Barrier block layout (byte offsets from off_bar).
constexpr uint32_t kBarWFull = 0;
constexpr uint32_t kBarWEmpty = kBarWFull + 8 * kMaxWStages;
constexpr uint32_t kBarAFull = kBarWEmpty + 8 * kMaxWStages;       // [kASlots]
constexpr uint32_t kBarAEmpty = kBarAFull + 8 * kASlots;            // [kASlots]
constexpr uint32_t kBarBReady = kBarAEmpty + 8 * kASlots;
constexpr uint32_t kBarDFull = kBarBReady + 8;                      // one arrival per issuer
constexpr uint32_t kWords = kBarDFull + 8;                          // uint32 scratch after barriers
// words: [0] tmem base, [1] abort, [2] bit mask of written accumulators,
// [3] band count, [4 + 2i] max|x| bits of activation row i, [5 + 2i] its
// band-B maximum, [20 + i] its count of nonzero elements below the band
// threshold, [28 + i] its sum of |x| (fp32)
constexpr uint32_t kWordsCount = 40;
constexpr uint32_t kBarBytes = kWords + kWordsCount * 4;

using namespace mma;

// kStageItems: activation words a staging thread takes per batch (see the
// staging warps).
template <bool SWIGLU, int kStageItems>
__global__ void __launch_bounds__(kThreads, 1)
k_tern_mma(const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_u, const MmaParams p)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *gbase = smem_raw + (base - raw);

    const uint32_t wbuf = base;
    const uint32_t bbuf = base + p.off_b;
    float *red = reinterpret_cast<float *>(gbase + p.off_red);   // [split][128][16]: pair (hi[8], lo[8]) per row
    float *xch = reinterpret_cast<float *>(gbase + p.off_xch);   // [64][8]
    const uint32_t bars = base + p.off_bar;
    uint32_t *words = reinterpret_cast<uint32_t *>(gbase + p.off_bar + kWords);
    volatile uint32_t *abort_flag = words + 1;
    uint32_t *xmax = words + 4;  // [2i], [2i + 1]: max |x| and band-B max (fp32 bits) of activation row i
    uint32_t *n_small = words + 20;
    float *sum_abs = reinterpret_cast<float *>(words + 28);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int split = p.split;
    const int rank = (int)(blockIdx.x % (unsigned)split);
    const int tile = (int)(blockIdx.x / (unsigned)split);
    const int st0 = rank * p.per_st;
    const int st1 = min(p.total_st, st0 + p.per_st);
    const int n_st = max(0, st1 - st0);
    const int n_chunks = n_st * (kStageWords / kChunkWords);  // 4 chunks per stage
    const int n_wst = p.n_wst;
    const int row0 = SWIGLU ? tile * 64 : tile * 128;
    const int m = p.m;

    auto issue = [&](int s) {
        const int slot = s % n_wst;
        const uint32_t dst = wbuf + slot * kStageBytes;
        const uint32_t full = bars + kBarWFull + 8 * slot;
        const int c0 = (st0 + s) * kStageWords;
        ptx::mbar_arrive_expect_tx(full, kStageBytes);
        if constexpr (SWIGLU) {
            ptx::tma_load_2d(dst, &tm_g, c0, row0, full);
            ptx::tma_load_2d(dst + kStageBytes / 2, &tm_u, c0, row0, full);
        } else {
            ptx::tma_load_2d(dst, &tm_g, c0, row0, full);
        }
    };

    // ---- prologue: barriers, first weight copies, tensor memory
    int issued = 0;
    if (tid == 0) {
        for (int s = 0; s < n_wst; ++s) {
            ptx::mbar_init(bars + kBarWFull + 8 * s, 1);
            ptx::mbar_init(bars + kBarWEmpty + 8 * s, 4);  // the four warps of the group that read it
        }
        for (int s = 0; s < kASlots; ++s) {
            ptx::mbar_init(bars + kBarAFull + 8 * s, 4);   // the four warps that wrote it
            ptx::mbar_init(bars + kBarAEmpty + 8 * s, kIssuers);
        }
        ptx::mbar_init(bars + kBarBReady, kStagers);
        ptx::mbar_init(bars + kBarDFull, kIssuers);
        for (int j = 1; j < (int)kWordsCount; ++j) words[j] = 0u;
        ptx::fence_proxy_async_smem();
        if (n_st > 0) {
            ptx::prefetch_tmap(&tm_g);
            if (SWIGLU) ptx::prefetch_tmap(&tm_u);
            for (; issued < n_st && issued < n_wst; ++issued) issue(issued);
        }
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
    const Waiter waiter(abort_flag, &g_mma_error, p.wait_limit);

    if (warp == 0) {
        // ----------------------------------------------------------- producer
        if (lane == 0) {
            for (; issued < n_st; ++issued) {
                const int slot = issued % n_wst;
                if (!waiter.wait(bars + kBarWEmpty + 8 * slot, ((issued / n_wst) - 1) & 1)) break;
                issue(issued);
            }
            // every issued copy must land before the CTA may exit
            for (int s = (issued > n_wst ? issued - n_wst : 0); s < issued; ++s)
                drain_wait(bars + kBarWFull + 8 * (s % n_wst), (s / n_wst) & 1, &g_mma_error);
        }
    } else if (warp <= kStagerWarps) {
        // ------------------------------------------------- B operand staging
        // Only these warps read data the previous grid may have written (the
        // activations), so only they wait for it; every MMA waits for b_ready.
        ptx::grid_dep_wait();
        const int st_tid = tid - 32;
        const int n_words = n_st * kStageWords;
        const int k0 = st0 * kStageWords * 16;
        const int n_items = m * n_words;  // (activation row, word) pairs with data
        // Items are processed in batches of kStageItems per thread: all loads of
        // a batch are issued before any is used, so a batch costs one memory
        // latency.  Small problems (n_items <= kStagers * kStageItems) keep
        // their activations in registers across the three passes.  The host
        // takes kStageItems = 1 when every item of the CTA fits one batch of
        // one per thread, else 4: each pass then runs a quarter of the code,
        // which a CTA executes once, with cold instruction caches.
        uint4 xa[kStageItems], xb[kStageItems];
        const bool resident = n_items <= kStagers * kStageItems;
        auto load_batch = [&](int first) {
#pragma unroll
            for (int t = 0; t < kStageItems; ++t) {
                const int item = first + t * kStagers;
                xa[t] = make_uint4(0, 0, 0, 0);
                xb[t] = make_uint4(0, 0, 0, 0);
                if (item < n_items) {
                    const int mm = item / n_words, wi = item - mm * n_words;
                    const int kk = k0 + 16 * wi;
                    if (kk < p.k) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (size_t)mm * p.k + kk);
                        xa[t] = src[0];
                        xb[t] = src[1];
                    }
                }
            }
        };
        // The two statistics passes reduce within each warp first and make one
        // shared-memory atomic per warp: a warp's 32 items at a given t are 32
        // consecutive words of one activation row (n_words is a multiple of
        // 32), and every thread takes the same number of turns, past n_items
        // with zeros.
        for (int base_i = 0; base_i < n_items; base_i += kStagers * kStageItems) {  // max |x| per row
            const int first = base_i + st_tid;
            load_batch(first);
#pragma unroll
            for (int t = 0; t < kStageItems; ++t) {
                const int item = first + t * kStagers;
                const uint32_t v = __reduce_max_sync(0xFFFFFFFFu, item < n_items ? max_abs16(xa[t], xb[t]) : 0u);
                const int item0 = item - lane;
                if (lane == 0 && item0 < n_items) atomicMax(&xmax[2 * (item0 / n_words)], v);
            }
        }
        ptx::named_bar_sync(3, kStagers);
        for (int base_i = 0; base_i < n_items; base_i += kStagers * kStageItems) {  // band B of each row
            const int first = base_i + st_tid;
            if (!resident) load_batch(first);
#pragma unroll
            for (int t = 0; t < kStageItems; ++t) {
                const int item = first + t * kStagers;
                const int item0 = item - lane;
                const int mm = item0 < n_items ? item0 / n_words : 0;
                const uint32_t tb2 = band_threshold2(xmax[2 * mm]);
                uint32_t n = 0, mb = 0;
                float sabs = 0.f;
                if (item < n_items) {
                    band_stats16(xa[t], xb[t], tb2, n, sabs);
                    mb = max_abs16_below(xa[t], xb[t], tb2);
                }
                mb = __reduce_max_sync(0xFFFFFFFFu, mb);
                n = __reduce_add_sync(0xFFFFFFFFu, n);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sabs += __shfl_xor_sync(0xFFFFFFFFu, sabs, o);
                if (lane == 0 && item0 < n_items) {
                    atomicMax(&xmax[2 * mm + 1], mb);
                    atomicAdd(&n_small[mm], n);
                    atomicAdd(&sum_abs[mm], sabs);
                }
            }
        }
        ptx::named_bar_sync(3, kStagers);
        // one or two bands for every row of this CTA's K range (need_two_bands)
        if (st_tid < m && need_two_bands(xmax[2 * st_tid], n_small[st_tid], sum_abs[st_tid])) atomicOr(&words[3], 1u);
        ptx::named_bar_sync(3, kStagers);
        const int bands = words[3] != 0u ? 2 : 1;
        const uint32_t wbytes = b_block_bytes(m, bands);
        for (int first = st_tid; first < n_items; first += kStagers * kStageItems) {  // e4m3 pieces
            if (!resident) load_batch(first);
#pragma unroll
            for (int t = 0; t < kStageItems; ++t) {
                const int item = first + t * kStagers;
                if (item >= n_items) break;
                const int mm = item / n_words, wi = item - mm * n_words;
                const uint32_t at = bbuf + (uint32_t)wi * wbytes + 32u * (uint32_t)(bands * mm);
                const float sca = exp2i(row_scale_exp(xmax[2 * mm]));
                if (bands == 2) {
                    uint4 rows[4];
                    split_word2(xa[t], xb[t], sca, exp2i(row_scale_exp(xmax[2 * mm + 1])), band_threshold2(xmax[2 * mm]),
                                rows);
#pragma unroll
                    for (int r = 0; r < 4; ++r) ptx::sts128(at + 16u * (uint32_t)r, rows[r]);
                } else {
                    uint4 rows[2];
                    split_word1(xa[t], xb[t], sca, rows);
                    ptx::sts128(at, rows[0]);
                    ptx::sts128(at + 16u, rows[1]);
                }
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(bars + kBarBReady);
        // ------------------------------------------------------- MMA issue
        // Issuer k takes the K=32 steps 4k..4k+3 of every stage (16 steps of
        // two words each) into its own accumulator D[k].
        const int k_iss = warp - 1;
        const int n_mma = mma_n(m, bands);
        const uint32_t idesc = idesc_n(n_mma);
        if (lane == 0) {
            bool ok = waiter.wait(bars + kBarBReady, 0);  // all staging warps are done
            const uint32_t d = tmem + kDCol + (uint32_t)(n_mma * k_iss);
            for (int st = 0; st < n_st && ok; ++st) {
                const int slot = st % kASlots;
                if (!waiter.wait(bars + kBarAFull + 8 * slot, (st / kASlots) & 1)) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int step = 4 * k_iss + t;               // K=32 step within the stage
                    const int wi = st * kStageWords + 2 * step;   // its first word
                    ptx::mma_ts_f8f6f4(d, tmem + (uint32_t)(slot * 128 + step * 8),
                                       b_desc_lbo(bbuf + (uint32_t)wi * wbytes, wbytes), idesc,
                                       (st | t) != 0 ? 1u : 0u);
                }
                ptx::mma_commit(bars + kBarAEmpty + 8 * slot);
                if (st == 0) atomicOr(&words[2], 1u << k_iss);  // accumulator written
            }
            ptx::mma_commit(bars + kBarDFull);  // arrives when this issuer's MMAs are done
        }
    } else {
        // ----------------------------------------------------------- decoders
        // Warpgroup g decodes every other stage; thread i owns row i (TMEM lane
        // i).  A stage is 32 words per row: four chunks of 8 words, each
        // stored to 32 columns of the stage's TMEM slot.  Only lane 0 polls
        // barriers; the warp follows it.
        const int g = (warp - kFirstDecWarp) >> 2;
        const int quad = warp & 3;                  // TMEM lane quadrant this warp may touch
        const int i = quad * 32 + lane;             // weight row within the tile == TMEM lane
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        const uint32_t row_addr = wbuf + (uint32_t)i * 128u;
        for (int st = g; st < n_st; st += 2) {
            const int wslot = st % n_wst;
            const int aslot = st % kASlots;
            uint32_t ok = 1u;
            if (lane == 0) {
                ok = waiter.wait(bars + kBarWFull + 8 * wslot, (st / n_wst) & 1) ? 1u : 0u;
                if (ok && st >= kASlots) ok = waiter.wait(bars + kBarAEmpty + 8 * aslot, ((st / kASlots) - 1) & 1) ? 1u : 0u;
            }
            if (__shfl_sync(0xFFFFFFFFu, ok, 0) == 0u) break;
            ptx::tc_fence_after();
            const uint32_t srow = row_addr + (uint32_t)wslot * kStageBytes;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                const uint4 v0 = ptx::lds128(srow + ((uint32_t)((2 * c) ^ (i & 7)) << 4));
                const uint4 v1 = ptx::lds128(srow + ((uint32_t)((2 * c + 1) ^ (i & 7)) << 4));
                uint32_t r[32];
                decode8(v0, v1, r);
                ptx::tmem_st_32x32b_x32(tmem + lane_addr + (uint32_t)(aslot * 128 + c * 32), r);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bars + kBarWEmpty + 8 * wslot);  // stage read: ring slot free
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bars + kBarAFull + 8 * aslot);   // my 32 rows are in TMEM
        }
    }

    // ------------------------------------------------------------- epilogue
    // The CTA barrier orders the staging warps' per-row scales (xmax) before
    // the epilogue reads them.
    __syncwarp();
    __syncthreads();
    // per activation row, this rank's sum: plain fp32 with one band, an
    // unevaluated pair (acc_pair) with two, whose terms, and then the ranks'
    // partials, may cancel at very different magnitudes
    float acc[8], acc_lo[8];
#pragma unroll
    for (int n = 0; n < 8; ++n) acc[n] = acc_lo[n] = 0.f;
    const bool epi = (warp >= kFirstDecWarp && warp < kFirstDecWarp + 4);  // warpgroup 0 reads D
    const int quad = warp & 3;
    const int i = quad * 32 + lane;
    if (epi && n_chunks > 0) {
        const int bands = words[3] != 0u ? 2 : 1;
        const int n_mma = mma_n(m, bands);
        if (waiter.wait(bars + kBarDFull, 0)) {
            ptx::tc_fence_after();
            const uint32_t written = words[2];
            const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16) + kDCol;
            // Sums the 16-column group at `col` of every written accumulator
            // (the same bands and scales: plain fp32 adds).
            auto sum_group = [&](uint32_t col, float (&dsum)[16]) {
#pragma unroll
                for (int q = 0; q < 16; ++q) dsum[q] = 0.f;
                for (int a = 0; a < kIssuers; ++a) {
                    if (!((written >> a) & 1u)) continue;
                    uint32_t d[16];
                    ptx::tmem_ld_32x32b_x16(lane_base + (uint32_t)(n_mma * a) + col, d);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 16; ++q) dsum[q] += __uint_as_float(d[q]);
                }
            };
            // each row's band terms, at their scales (hi 2^-s, lo 2^-(s+4)
            // of each band), go into its pair
            if (bands == 1) {  // column 2i + b of row i: hi, lo
                float dsum[16];
                sum_group(0u, dsum);
                // one band: each row's sum is within 2^-24 of its sum |x|
                // already, so it stays a plain fp32 sum (acc_lo stays zero)
#pragma unroll
                for (int mm = 0; mm < 8; ++mm) {
                    if (mm < m) {
                        const int sa = row_scale_exp(xmax[2 * mm]);
                        acc[mm] = fmaf(dsum[2 * mm + 1], exp2i(-sa - 4), dsum[2 * mm] * exp2i(-sa));
                    }
                }
            } else {  // column 4i + b of row i: hi_A, lo_A, hi_B, lo_B
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (4 * h >= m) break;
                    float dsum[16];
                    sum_group(16u * (uint32_t)h, dsum);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int mm = 4 * h + r;
                        if (mm < m) {
                            const int sa = row_scale_exp(xmax[2 * mm]), sb = row_scale_exp(xmax[2 * mm + 1]);
                            acc_pair(acc[mm], acc_lo[mm], dsum[4 * r] * exp2i(-sa));
                            acc_pair(acc[mm], acc_lo[mm], dsum[4 * r + 1] * exp2i(-sa - 4));
                            acc_pair(acc[mm], acc_lo[mm], dsum[4 * r + 2] * exp2i(-sb));
                            acc_pair(acc[mm], acc_lo[mm], dsum[4 * r + 3] * exp2i(-sb - 4));
                        }
                    }
                }
            }
        }
    }
    ptx::tc_fence_before();
    if (split > 1) {
        // every rank pushes its partial into rank 0's buffer slot [rank]; one
        // cluster barrier; rank 0 sums the slots in rank order
        if (epi) {
            const uint32_t dst = ptx::mapa(ptx::smem_u32(red + ((size_t)rank * 128 + i) * 16), 0u);
            ptx::st_cluster_v4(dst, acc[0], acc[1], acc[2], acc[3]);
            ptx::st_cluster_v4(dst + 16u, acc[4], acc[5], acc[6], acc[7]);
            ptx::st_cluster_v4(dst + 32u, acc_lo[0], acc_lo[1], acc_lo[2], acc_lo[3]);
            ptx::st_cluster_v4(dst + 48u, acc_lo[4], acc_lo[5], acc_lo[6], acc_lo[7]);
        }
        ptx::cluster_arrive();
        ptx::cluster_wait();
        if (epi && rank == 0) {
#pragma unroll
            for (int n = 0; n < 8; ++n) acc[n] = acc_lo[n] = 0.f;
            // plain fp32 adds while every rank had one band (its lo parts
            // are zero); exact pairs once a rank took two
            bool pairs = false;
            for (int r = 0; r < split; ++r) {
                const float *v = red + ((size_t)r * 128 + i) * 16;
#pragma unroll
                for (int n = 0; n < 8; ++n) pairs = pairs || v[8 + n] != 0.f;
            }
            for (int r = 0; r < split; ++r) {
                const float *v = red + ((size_t)r * 128 + i) * 16;
                if (pairs) {
#pragma unroll
                    for (int n = 0; n < 8; ++n) {
                        acc_pair(acc[n], acc_lo[n], v[n]);
                        acc_pair(acc[n], acc_lo[n], v[8 + n]);
                    }
                } else {
#pragma unroll
                    for (int n = 0; n < 8; ++n) acc[n] += v[n];
                }
            }
        }
    }
#pragma unroll
    for (int n = 0; n < 8; ++n) acc[n] = __fadd_rn(acc[n], acc_lo[n]);
    if (rank == 0 && epi) {
        if constexpr (SWIGLU) {
            const int r = row0 + (i & 63);
            if (i >= 64 && r < p.rows) {
                const float su = p.scale_u[r];
#pragma unroll
                for (int n = 0; n < 8; ++n) xch[(i - 64) * 8 + n] = su * (0.5f * acc[n]);
            }
            ptx::named_bar_sync(1, 128);
            if (i < 64 && r < p.rows) {
                const float sg = p.scale_g[r];
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    if (n < m) {
                        const float gv = sg * (0.5f * acc[n]);
                        p.y[(size_t)n * p.rows + r] = silu_f(gv) * xch[i * 8 + n];
                    }
                }
            }
        } else {
            const int r = row0 + i;
            if (r < p.rows) {
                const float sc = p.scale_g[r];
#pragma unroll
                for (int n = 0; n < 8; ++n)
                    if (n < m) p.y[(size_t)n * p.rows + r] = sc * (0.5f * acc[n]);
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        // On an abort path MMAs may still be in flight: wait (bounded) for
        // their commits before the tensor memory is released.
        if (lane == 0) drain_wait(bars + kBarDFull, 0, &g_mma_error);
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side

template <bool SWIGLU>
tern_status launch_mma(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int m, float *y,
                       cudaStream_t stream)
{
    const int rows = g->rows, k = g->k, kw = k / 16;
    const int tile_rows = SWIGLU ? 64 : 128;
    const int tiles = (rows + tile_rows - 1) / tile_rows;
    const int total_st = (kw + kStageWords - 1) / kStageWords;
    const int sms = sm_count();

    // Split K over a cluster while the CTAs still fit the SMs and each rank
    // keeps at least four stages.  Measured one call at a time on the
    // decode shapes: 1024x4096 at split 2 / 4 / 8 took 7.7 / 8.3 / 11.3 us,
    // 4096x4096 at 2 / 4 took 8.0 / 9.0 us, and the 4096x12288 down
    // projection ran faster at 4 than at 2.  Each rank pays its own prologue,
    // statistics passes and cluster exchange; below four stages that costs
    // more than the wider weight stream gains.
    int split = 1;
    while (split < 8 && tiles * split * 2 <= sms && split * 2 * 4 <= total_st) split *= 2;
    const uint32_t wbytes = b_block_bytes(m, 2);  // room for two bands
    int per_st = 0, n_wst = 0;
    for (;;) {
        per_st = total_st > 0 ? (total_st + split - 1) / split : 0;
        // split-K partials (a pair of 8 per row per rank), SwiGLU exchange, barriers
        const uint32_t misc = (uint32_t)split * 128 * 16 * 4 + 64 * 8 * 4 + kBarBytes + 64;
        const uint32_t fixed = 1024 + (uint32_t)per_st * kStageWords * wbytes + kBPad + misc;
        n_wst = fixed < (uint32_t)kSmemLimit ? (int)((kSmemLimit - fixed) / kStageBytes) : 0;
        if (n_wst > kMaxWStages) n_wst = kMaxWStages;
        if (n_wst > per_st && per_st >= 1) n_wst = per_st < 2 ? 2 : per_st;  // no deeper than the work
        // Even depth: the two decoder warpgroups take alternate stages, so a
        // ring slot is then always reused by the group that last used it and
        // a phase-parity wait never runs two phases ahead of its barrier.
        n_wst &= ~1;
        if (n_wst >= 2 || split >= 8) break;
        split *= 2;
    }
    if (n_wst < 2) return TERN_ERR_SHAPE;

    MmaParams prm;
    prm.scale_g = g->scale;
    prm.scale_u = SWIGLU ? u->scale : nullptr;
    prm.x = x;
    prm.y = y;
    prm.rows = rows;
    prm.k = k;
    prm.m = m;
    prm.total_st = total_st;
    prm.per_st = per_st;
    prm.split = split;
    prm.n_wst = n_wst;
    prm.wait_limit = wait_limit();
    prm.off_b = (uint32_t)n_wst * kStageBytes;
    prm.off_red = prm.off_b + (uint32_t)per_st * kStageWords * wbytes + kBPad;
    prm.off_xch = prm.off_red + (uint32_t)split * 128 * 16 * 4;
    prm.off_bar = prm.off_xch + 64 * 8 * 4;
    uint32_t smem = 1024 + prm.off_bar + kBarBytes;
    if (smem < kMinSmem) smem = kMinSmem;

    CUtensorMap tg, tu;
    std::memset(&tg, 0, sizeof(tg));
    std::memset(&tu, 0, sizeof(tu));
    if (kw > 0) {
        if (!make_code_map(&tg, g->codes, rows, kw, tile_rows)) return TERN_ERR_CUDA;
        if (SWIGLU && !make_code_map(&tu, u->codes, rows, kw, tile_rows)) return TERN_ERR_CUDA;
    }

    // staging batch: one activation word per thread when a CTA's words (its
    // K range, every activation row) fit the staging threads once
    const bool one_item = (long long)m * per_st * kStageWords <= kStagers;
    auto kern = one_item ? k_tern_mma<SWIGLU, 1> : k_tern_mma<SWIGLU, 4>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return TERN_ERR_CUDA;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * split), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (split > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)split;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, kern, tg, tu, prm) != cudaSuccess) return TERN_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? TERN_OK : TERN_ERR_CUDA;
}

}  // namespace

namespace mma {

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiled encode_fn()
{
    static EncodeTiled fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    }
    return fn;
}

namespace {

// Encoded tensor maps by (codes, rows, kw, box_rows): a map depends on
// nothing else, so a reused key (the same matrix called again, or a new
// allocation at the same address with the same shape) reuses its map and the
// per-call host cost of a batch of resident weights is a table lookup.
struct MapKey {
    const uint32_t *codes;
    int rows, kw, box_rows;
    bool operator==(const MapKey &o) const
    {
        return codes == o.codes && rows == o.rows && kw == o.kw && box_rows == o.box_rows;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey &k) const
    {
        size_t h = std::hash<const void *>()(k.codes);
        h ^= ((size_t)k.rows * 0x9E3779B97F4A7C15ull) + ((size_t)k.kw << 20) + (size_t)k.box_rows;
        return h;
    }
};
constexpr size_t kMapCacheMax = 8192;
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_map_cache;

}  // namespace

bool make_code_map(CUtensorMap *m, const uint32_t *codes, int rows, int kw, int box_rows)
{
    const MapKey key{codes, rows, kw, box_rows};
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto f = g_map_cache.find(key);
        if (f != g_map_cache.end()) {
            *m = f->second;
            return true;
        }
    }
    EncodeTiled fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kw, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kw * 4};
    const cuuint32_t box[2] = {(cuuint32_t)kStageWords, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t *>(codes), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_map_cache.size() >= kMapCacheMax) g_map_cache.clear();
    g_map_cache.emplace(key, *m);
    return true;
}

}  // namespace mma

tern_status gemm_mma(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int m, float *y,
                     cudaStream_t s)
{
    if (m < 1 || m > 8) return TERN_ERR_M_RANGE;
    return u ? launch_mma<true>(g, u, x, m, y, s) : launch_mma<false>(g, nullptr, x, m, y, s);
}

tern_status take_mma_error()
{
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_mma_error, sizeof(v)) != cudaSuccess) return TERN_ERR_CUDA;
    if (v != 0u) {
        if (cudaMemcpyToSymbol(g_mma_error, &z, sizeof(z)) != cudaSuccess) return TERN_ERR_CUDA;
        return TERN_ERR_TIMEOUT;
    }
    return TERN_OK;
}

}  // namespace tern
