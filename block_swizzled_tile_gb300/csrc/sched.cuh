// Device tile scheduler: the task index -> output tile mapping of
// GemmIdentityBlockSwizzle ("Block Scheduler Code Explained", sections 4.3
// GetCoreLoops, 4.4 GetBatchIdx, 4.5 GetBlockCoord, 4.6 GetActualBlockShape,
// 5 Scheduling Policies, 6 DynamicGemmIdentityBlockSwizzle), with the offset
// and direction chosen at run time as in the dynamic variant.
//
// Differences from the page's code, none of which changes the map:
//  * the offset is clamped to the number of tile-rows (Zn) / tile-columns
//    (Nz).  With SwizzleOffset >= loopsM there is a single window whose height
//    is loopsM, so the map is the same; the clamp keeps offset * loops inside
//    32 bits for any offset the caller passes.
//  * the Nz branch, elided on the page, is the transpose of Zn: windows of
//    SwizzleOffset tile-columns, n fastest inside a window, m reversed on odd
//    windows (the page's prose divides the grid by columns for Nz and has the
//    snake reverse the index along the window).
#pragma once
#include <cstdint>

namespace bst {

struct SwizzleSched {
    uint32_t M, N;            // problem extent (elements)
    uint32_t tile_m, tile_n;  // tile extent (elements)
    uint32_t loops_m, loops_n;
    uint32_t offset;          // SwizzleOffset after the clamp
    uint32_t direction;       // 0 Zn, 1 Nz

    __host__ __device__ static uint32_t ceil_div(uint32_t a, uint32_t b) { return (a + b - 1) / b; }

    // constructor + Update (sections 4.1, 4.2): loop counts by ceiling division
    __host__ __device__ void update(uint32_t M_, uint32_t N_, uint32_t tm, uint32_t tn, uint32_t swz_offset,
                                    uint32_t swz_dir) {
        M = M_;
        N = N_;
        tile_m = tm;
        tile_n = tn;
        loops_m = ceil_div(M_, tm);
        loops_n = ceil_div(N_, tn);
        direction = swz_dir;
        const uint32_t lim = swz_dir == 0 ? loops_m : loops_n;
        offset = swz_offset < lim ? swz_offset : (lim > 0 ? lim : 1);
    }

    __host__ __device__ uint32_t core_loops() const { return loops_m * loops_n; }       // section 4.3
    __host__ __device__ uint32_t batch_idx(uint32_t t) const { return t / core_loops(); }  // section 4.4

    // section 4.5
    __host__ __device__ void block_coord(uint32_t t, uint32_t& m, uint32_t& n) const {
        const uint32_t inner = t % core_loops();
        const uint32_t S = offset;
        if (direction == 0) {
            const uint32_t per_window = S * loops_n;
            const uint32_t window = inner / per_window;
            const uint32_t pos = inner - window * per_window;
            const uint32_t last = ceil_div(loops_m, S) - 1;
            const uint32_t h = window == last ? loops_m - S * window : S;
            m = window * S + pos % h;
            n = pos / h;
            if (window & 1u) n = loops_n - 1 - n;
        } else {
            const uint32_t per_window = S * loops_m;
            const uint32_t window = inner / per_window;
            const uint32_t pos = inner - window * per_window;
            const uint32_t last = ceil_div(loops_n, S) - 1;
            const uint32_t w = window == last ? loops_n - S * window : S;
            n = window * S + pos % w;
            m = pos / w;
            if (window & 1u) m = loops_m - 1 - m;
        }
    }

    // section 4.6 (kActual is always the whole K)
    __host__ __device__ void actual_shape(uint32_t m, uint32_t n, uint32_t& m_act, uint32_t& n_act) const {
        m_act = m == loops_m - 1 ? M - m * tile_m : tile_m;
        n_act = n == loops_n - 1 ? N - n * tile_n : tile_n;
    }
};

// Grouped slice-M: per-group tile offsets (group-major task numbering) and row
// offsets, as exclusive prefix sums of the group sizes.  Filled once per CTA
// in shared memory; `find` maps a task to its group by binary search.
// Unsigned 32-bit division by a divisor fixed before the launch.  The host
// picks s = ceil(log2 d) and m = ceil(2^(32+s) / d) - 2^32, and then
// n / d = (umulhi(n, m) + n) >> s for every 32-bit n (the round-up method of
// Granlund and Montgomery, "Division by invariant integers using
// multiplication"): a multiply and a shift on the device instead of the
// ~25-instruction dependent sequence of a division by a run-time value,
// which a single scheduling thread pays in full.
struct FastDiv {
    uint32_t d, m, s;

    static FastDiv make(uint32_t d_) {
        FastDiv f;
        f.d = d_ ? d_ : 1u;
        f.s = 0;
        while ((1ull << f.s) < f.d) ++f.s;
        const unsigned __int128 one = 1;
        f.m = static_cast<uint32_t>(((one << (32 + f.s)) + f.d - 1) / f.d - (one << 32));
        return f;
    }
#ifdef __CUDACC__
    __device__ __forceinline__ uint32_t div(uint32_t n) const {
        return static_cast<uint32_t>((static_cast<uint64_t>(__umulhi(n, m)) + n) >> s);
    }
#endif
};

// The scheduler of a plain or batched problem with everything that does not
// depend on the task index computed on the host: the same map as
// SwizzleSched (sections 4.1-4.6: ceiling-division loop counts, the clamped
// SwizzleOffset, windows, snake, actual block shape), with its divisions by
// the core-loop count, the window size and the window height done through
// FastDiv.
struct PlainSched {
    uint32_t M, N, tile_m, tile_n, loops_m, loops_n;
    uint32_t S, dir;
    uint32_t last;            // index of the last window
    FastDiv core;             // loops_m * loops_n: batch index and task within the batch
    FastDiv per_window;       // S * loops_n (Zn) or S * loops_m (Nz)
    FastDiv win;              // S: tile rows (Zn) / columns (Nz) of a full window
    FastDiv win_last;         // the same for the last, possibly narrower window

    void init(uint32_t M_, uint32_t N_, uint32_t tm, uint32_t tn, uint32_t swz_offset, uint32_t swz_dir) {
        SwizzleSched r;
        r.update(M_, N_, tm, tn, swz_offset, swz_dir);
        M = M_; N = N_; tile_m = tm; tile_n = tn;
        loops_m = r.loops_m; loops_n = r.loops_n;
        S = r.offset; dir = swz_dir;
        const uint32_t lim = dir == 0 ? loops_m : loops_n;
        last = lim ? (lim + S - 1) / S - 1 : 0;
        core = FastDiv::make(loops_m * loops_n);
        per_window = FastDiv::make(S * (dir == 0 ? loops_n : loops_m));
        win = FastDiv::make(S);
        win_last = FastDiv::make(lim ? lim - S * last : 1);
    }
#ifdef __CUDACC__
    __device__ __forceinline__ void coord(uint32_t t, uint32_t& batch, uint32_t& m, uint32_t& n, uint32_t& m_act,
                                          uint32_t& n_act) const {
        batch = core.div(t);
        const uint32_t inner = t - batch * core.d;
        const uint32_t window = per_window.div(inner);
        const uint32_t pos = inner - window * per_window.d;
        const bool is_last = window == last;
        const FastDiv w{is_last ? win_last.d : win.d, is_last ? win_last.m : win.m, is_last ? win_last.s : win.s};
        const uint32_t q = w.div(pos);
        const uint32_t rem = pos - q * w.d;
        if (dir == 0) {
            m = window * S + rem;
            n = q;
            if (window & 1u) n = loops_n - 1 - n;
        } else {
            n = window * S + rem;
            m = q;
            if (window & 1u) m = loops_m - 1 - m;
        }
        m_act = m == loops_m - 1 ? M - m * tile_m : tile_m;
        n_act = n == loops_n - 1 ? N - n * tile_n : tile_n;
    }
#endif
};

struct GroupTable {
    uint32_t* tile_off;   // [G+1]
    uint32_t* row_off;    // [G+1]
    uint32_t G;

    __device__ uint32_t find(uint32_t t) const {
        uint32_t lo = 0, hi = G;  // invariant: tile_off[lo] <= t < tile_off[hi]
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (tile_off[mid] <= t) lo = mid; else hi = mid;
        }
        return lo;
    }
};

}  // namespace bst
