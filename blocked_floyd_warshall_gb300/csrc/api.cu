// C ABI of libbsmooth: argument checks, dispatch to the kernels, the small
// per-device buffer used by the feasibility count and the input check, launch
// counting and the optional per-phase event profile.
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/bsmooth.h"
#include "bs_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;

// A side stream and three events for the look-ahead schedule.  A call holds
// one exclusively while it enqueues, so concurrent callers never share events.
struct SideCtx {
    cudaStream_t side = nullptr;
    cudaEvent_t main_done[2] = {nullptr, nullptr};   // on the caller's stream, by round parity
    cudaEvent_t side_done = nullptr;                 // on the side stream
    cudaEvent_t next_done = nullptr;                 // on the side stream, after NEXT(K)
    cudaEvent_t near_done = nullptr;                 // on the side stream, after NEAR2(K)
};

struct DeviceState {
    bool ready = false;                   // kernel attributes set
    int sms = 0;                          // multiprocessor count
    unsigned long long* scratch = nullptr;  // [0] count, [1] validation flags
    std::vector<SideCtx> free_side;       // idle look-ahead contexts
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<long long> g_launches{0};

// ---- profiling ------------------------------------------------------------

struct ProfRec {
    cudaEvent_t a, b;
    int phase;
};
constexpr size_t kMaxProf = 1u << 16;
std::mutex g_prof_mu;
bool g_prof_on = false;
bool g_prof_overflow = false;
std::vector<ProfRec> g_prof;
thread_local cudaEvent_t t_pending = nullptr;

cudaError_t device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = bs::blocked_setup(false);
        if (e == cudaSuccess) e = bs::blocked_setup(true);
        if (e == cudaSuccess) e = bs::fused_setup(false);
        if (e == cudaSuccess) e = bs::fused_setup(true);
        if (e != cudaSuccess) return e;
        d.ready = true;
    }
    *out = &d;
    return cudaSuccess;
}

cudaError_t device_scratch(unsigned long long** out) {
    DeviceState* d = nullptr;
    cudaError_t e = device_state(&d);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!d->scratch) {
        e = cudaMalloc(reinterpret_cast<void**>(&d->scratch), 2 * sizeof(unsigned long long));
        if (e != cudaSuccess) {
            d->scratch = nullptr;
            return e;
        }
    }
    *out = d->scratch;
    return cudaSuccess;
}

cudaError_t acquire_side(DeviceState* d, SideCtx* out) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!d->free_side.empty()) {
            *out = d->free_side.back();
            d->free_side.pop_back();
            return cudaSuccess;
        }
    }
    // Highest priority: the work distributor then hands the next free SM slot
    // to phases 1 and 2 of round K+1 instead of to more tiles of round K.
    SideCtx c;
    int lo = 0, hi = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&c.side, cudaStreamNonBlocking, hi);
    for (cudaEvent_t* ev :
         {&c.main_done[0], &c.main_done[1], &c.side_done, &c.next_done, &c.near_done})
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        for (cudaEvent_t ev : {c.main_done[0], c.main_done[1], c.side_done, c.next_done, c.near_done})
            if (ev) cudaEventDestroy(ev);
        if (c.side) cudaStreamDestroy(c.side);
        return e;
    }
    *out = c;
    return cudaSuccess;
}

void release_side(DeviceState* d, const SideCtx& c) {
    std::lock_guard<std::mutex> lk(g_mu);
    d->free_side.push_back(c);
}

// Block rows from which 128-wide tiles take block rounds in pairs.  Measured
// (ms, single rounds against pairs): n = 16384 759.6 / 734.9, n = 12288
// 324.8 / 314.5, n = 8192 on 128-wide tiles 98.5 / 95.2; upper bound alone
// n = 16384 247.1 / 241.6, n = 8192 32.0 / 31.5, n = 4096 (32 block rows)
// 4.4-4.8 / 5.5: with few rows the side stream's chain per pair (two serial
// phase-1 closures among the rest) outlasts the pair's bulk.
constexpr int PAIRS_FROM = 48;
// 64-wide tiles take block rounds in pairs once a pair's bulk (REST2) holds
// at least this many tiles over the batch.  Measured (ms, one round per pass
// against pairs): n = 4096 (3600 tiles) 12.88 / 12.45, n = 6000 39.5 / 37.7,
// int32 n = 4096 13.65 / 13.26, 256 x n = 512 (4096) 6.22 / 6.01, symmetric
// 256 x n = 512 (2560) 3.76 / 3.69, symmetric n = 8192 (7750) 50.6 / 47.9;
// n = 3584 (2704) 8.79 / 8.53, symmetric n = 5120 (2926) 12.96 / 12.58,
// symmetric n = 6144 (4278) 21.97 / 21.10; at the threshold n = 3456 (2500)
// 7.90 / 7.90; below it n = 3000 (1849) 5.56 / 5.54, symmetric n = 4096
// (1830) 7.15 / 7.57, n = 2048 (784) 2.14 / 2.47, n = 1000 0.59 / 0.86.
constexpr double PAIRS_TILES_64 = 2500.0;

bool pairs_pay(const bs::Mats& m, int nb) {
    if (m.fb == bs::FB_LARGE) return nb >= PAIRS_FROM;
    const double r = nb - 4.0;
    const double rest2 = r <= 0 ? 0.0 : m.sym ? r * (r + 1) / 2 : r * r;
    return rest2 * m.batch >= PAIRS_TILES_64;
}

// Tile size for the blocked schedule: 128 x 128 from PAIRS_FROM block rows
// of 128 for general inputs (single matrices from n = 6017 on; symmetric
// inputs keep one round per pass) or once a block round's phase 3
// at 128 holds at least 9000 tiles over the batch, else 64 x 64; fp32 and
// int32 alike.  With 48 rows or more the 128-wide schedule takes block
// rounds in pairs and wins (ms, 64 against 128 in pairs: fp32 n = 6144
// 41.5 / 41.0, n = 8192 96.8 / 95.2, n = 10240 188.3 / 186.8; int32
// n = 6144 43.9 / 42.6, n = 8192 102.6 / 99.1; at n = 5120, 40 rows, one
// round per pass, 24.5 / 25.7).  Before pairs, measured on the
// GB300 (ms, 64 against 128): fp32 n = 4096 12.92 / 13.22, n = 6000 39.6 /
// 41.1, n = 8192 97.1 / 98.6, n = 10000 178.8 / 185.7, n = 12288 324.7 /
// 324.6, n = 16384 766.8 / 758.7; 64 molecules of n = 1024 12.24 / 12.40;
// int32 n = 3000 5.91 / 6.46, n = 6000 41.8 / 42.8, n = 8192 102.6 / 102.6,
// n = 16384 810.4 / 793.1.  The smaller tiles spread further over the SMs
// and keep the serial phase 1 short; the larger halve the block rounds.
// The upper bound alone takes 128 from 768 tiles: its 128-wide form has its
// k loop unrolled (n = 4096: 5.3 against 5.8 ms; n = 6000: 15.7 against
// 17.7 ms; n = 3000, 529 tiles: 3.3 against 2.6 ms).
int choose_tile(int n, int batch, int mode, bool bounds) {
    if (mode & BS_TILE_64) return bs::FB_SMALL;
    if (mode & (BS_TILE_128 | BS_PAIRED_ROUNDS)) return bs::FB_LARGE;   // pairs: 128 unless 64 is asked
    const double nb = (double)((n + bs::FB_LARGE - 1) / bs::FB_LARGE);
    if (bounds && !(mode & BS_SYMMETRIC) && nb >= PAIRS_FROM) return bs::FB_LARGE;   // in pairs
    const double from = bounds ? 9000.0 : 768.0;
    return (nb - 1) * (nb - 1) * batch >= from ? bs::FB_LARGE : bs::FB_SMALL;
}

// The blocked schedule.  Without look-ahead: for each block round K, phase 1,
// phase 2, phase 3 on `s`.  With look-ahead (nb >= 3), phase 3 of round K is
// split into NEXT(K), the tiles of block-row/column K+1, and REST(K), the
// others, and two streams run
//   side: NEXT(K), phase 1 and phase 2 of round K+1   (highest priority)
//   s   : REST(K)
// concurrently.  NEXT(K) waits for REST(K-1) (it rewrites tiles REST(K-1)
// reads as panels), REST(K) for phase 2 of round K.  REST(K) touches no tile
// the side stream reads or writes in the meantime: it reads block-row and
// -column K, which phase 2 of round K+1 does not write except tiles (K,K+1)
// and (K+1,K), which REST(K) does not read; it writes tiles outside
// block-rows and -columns K and K+1.  NEXT(K)'s short wave thus overlaps
// REST(K) instead of running alone (except with few rest tiles, see below).
// With 64-wide tiles and few rest tiles (see `merged` below) phase 3 of
// round K runs whole but for tile (K+1,K+1) (P3_ALL_OFF) on `s`, and phase 1
// of round K+1 on the side stream applies round K's update to that tile
// itself before closing it, so the two run side by side: phase 1 reads tiles
// (K+1,K) and (K,K+1), which phase 3 only reads too, and writes tile
// (K+1,K+1), which phase 3 leaves alone; phase 1 waits for phase 3 of round
// K-1 (which writes tile (K+1,K+1)), phase 2 of round K+1 for phase 3 of
// round K, and phase 3 of round K+1 for phase 2 of round K+1.  With
// symmetric inputs a last launch on `s` writes the lower triangle as the
// transpose of the upper one.
// Block rounds in pairs (K, K+1), K even (see pairs_pay for when).
// The bulk of the tiles -- outside block-rows and -columns K .. K+3 -- takes
// both rounds in one pass (P3_REST2, on `s`), so each is loaded and stored
// once per pair instead of once per round (n = 16384 without look-ahead:
// 777.9 -> 750.6 ms, same bits).  The side stream carries, per pair, what the
// next steps need first:
//   NEXT(K): block-row and -column K+1 take round K; phases 1 and 2 of K+1
//            -> event P (the pair's panels are final);
//   NEAR2(K): block-rows and -columns K+2, K+3 outside K, K+1 take both
//            rounds -> event N;
//   CORNER2: tiles (K+2,K), (K+3,K), (K,K+2), (K,K+3) take round K+1;
//   phases 1 and 2 of K+2; NEXT(K+2); phases 1 and 2 of K+3 -> event P;
// and `s`, after P: REST2(K); after N: PREV2, the rest of block-row and
// -column K outside K+1 .. K+3 takes round K+1 -> event M.  The side stream
// waits for M before NEAR2 of the next pair, whose tiles REST2(K) and PREV2
// update.  Side by side the two streams touch disjoint tiles: REST2(K)
// writes tiles outside block-rows and -columns K .. K+3 and reads rows and
// columns K, K+1 there; the side stream writes tiles of block-rows and
// -columns K+1 .. K+3 only and reads rows and columns K .. K+3.  PREV2
// rewrites tiles of block-row and -column K that REST2(K) and NEAR2(K) read
// as panels of round K, hence its two waits.  An odd last round runs alone
// at the end (P3_ALL).  With symmetric inputs every set keeps its tiles on
// and above the diagonal (the panels are stored on both sides as always)
// and the lower triangle is written at the end.
cudaError_t run_pairs(bool is_int, const bs::Mats& m, cudaStream_t s, int nb, SideCtx& c) {
    using namespace bs;
    // phases 1 and 2 of round 0 are on `s`
    cudaError_t e = cudaEventRecord(c.main_done[0], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c.side, c.main_done[0], 0);
    if (e == cudaSuccess) e = launch_phase3(is_int, m, 0, P3_NEXT, c.side);
    if (e == cudaSuccess) e = launch_phase1(is_int, m, 1, false, c.side);
    if (e == cudaSuccess) e = launch_phase2(is_int, m, 1, c.side);
    if (e == cudaSuccess) e = cudaEventRecord(c.next_done, c.side);
    int K = 0;
    for (; K + 1 < nb && e == cudaSuccess; K += 2) {
        e = cudaStreamWaitEvent(s, c.next_done, 0);
        if (e == cudaSuccess) e = launch_phase3(is_int, m, K, P3_REST2, s);
        if (e == cudaSuccess && K > 0) e = cudaStreamWaitEvent(c.side, c.main_done[0], 0);
        if (e == cudaSuccess) e = launch_phase3(is_int, m, K, P3_NEAR2, c.side);
        if (e == cudaSuccess) e = cudaEventRecord(c.near_done, c.side);
        if (e == cudaSuccess) e = launch_phase3(is_int, m, K + 1, P3_CORNER2, c.side);
        if (e == cudaSuccess && K + 2 < nb) e = launch_phase1(is_int, m, K + 2, false, c.side);
        if (e == cudaSuccess && K + 2 < nb) e = launch_phase2(is_int, m, K + 2, c.side);
        if (e == cudaSuccess && K + 3 < nb) {
            e = launch_phase3(is_int, m, K + 2, P3_NEXT, c.side);
            if (e == cudaSuccess) e = launch_phase1(is_int, m, K + 3, false, c.side);
            if (e == cudaSuccess) e = launch_phase2(is_int, m, K + 3, c.side);
            if (e == cudaSuccess) e = cudaEventRecord(c.next_done, c.side);
        }
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, c.near_done, 0);
        if (e == cudaSuccess) e = launch_phase3(is_int, m, K + 1, P3_PREV2, s);
        if (e == cudaSuccess) e = cudaEventRecord(c.main_done[0], s);
    }
    // always join the side stream back, on success or failure
    cudaError_t r = cudaEventRecord(c.side_done, c.side);
    if (r == cudaSuccess) r = cudaStreamWaitEvent(s, c.side_done, 0);
    if (e == cudaSuccess) e = r;
    if (e == cudaSuccess && K == nb - 1) e = launch_phase3(is_int, m, K, P3_ALL, s);
    if (e == cudaSuccess && m.sym) e = launch_mirror(is_int, m, s);
    return e;
}


cudaError_t run_blocked(bool is_int, const bs::Mats& m, cudaStream_t s, bool lookahead,
                        bool force_pairs, DeviceState* d) {
    const int nb = (m.n + m.fb - 1) / m.fb;
    cudaError_t e = bs::launch_phase1(is_int, m, 0, false, s);
    if (e == cudaSuccess) e = bs::launch_phase2(is_int, m, 0, s);
    if (e != cudaSuccess) return e;
    if (!lookahead || nb < 3) {
        for (int K = 0; K < nb && e == cudaSuccess; ++K) {
            e = bs::launch_phase3(is_int, m, K, bs::P3_ALL, s);
            if (e == cudaSuccess && K + 1 < nb) e = bs::launch_phase1(is_int, m, K + 1, false, s);
            if (e == cudaSuccess && K + 1 < nb) e = bs::launch_phase2(is_int, m, K + 1, s);
        }
        if (e == cudaSuccess && m.sym) e = bs::launch_mirror(is_int, m, s);
        return e;
    }
    SideCtx c;
    e = acquire_side(d, &c);
    if (e != cudaSuccess) return e;
    if (force_pairs || pairs_pay(m, nb)) {
        e = run_pairs(is_int, m, s, nb, c);
        release_side(d, c);
        return e;
    }
    // With fewer rest-of-round tiles than SMs, REST(K) would take the SMs
    // the moment it is ready and phase 1 of round K+1, on the critical path,
    // would wait for its CTAs to finish; REST(K) then waits for NEXT(K)
    // instead (which follows phase 2 of round K on the side stream), so
    // phase 1 is dispatched first.  With more, REST(K) is long enough that
    // starting it early pays more (measured).
    // A call captured into a CUDA graph takes the tight order at every size:
    // replayed, the stream priority did not keep REST(K) from delaying phase 1
    // (n = 1000: 0.72 -> 0.64 ms, n = 2048: 2.66 -> 2.42 ms replayed).
    const double rest_tiles = m.sym ? 0.5 * (nb - 2) * (nb - 1) : (double)(nb - 2) * (nb - 2);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
        (void)cudaGetLastError();
        cap = cudaStreamCaptureStatusNone;
    }
    const bool tight = cap == cudaStreamCaptureStatusActive || rest_tiles * m.batch < m.sms;
    // main_done[1] stands for "REST(-1)": everything enqueued on s so far.
    e = cudaEventRecord(c.main_done[1], s);
    bool forked = false;   // side work enqueued that s has not yet waited for
    auto rest = [&](int K, cudaEvent_t after) {
        cudaError_t r = cudaSuccess;
        if (after) r = cudaStreamWaitEvent(s, after, 0);
        if (r == cudaSuccess) r = bs::launch_phase3(is_int, m, K, bs::P3_REST, s);
        if (r == cudaSuccess) r = cudaEventRecord(c.main_done[K & 1], s);
        return r;
    };
    // 64-wide tiles, fewer rest tiles than half the SMs: the chain NEXT(K),
    // phases 1 and 2 of round K+1 is then the critical path, so NEXT(K) and
    // REST(K) become one launch without tile (K+1,K+1), beside phase 1 of
    // round K+1, which applies round K's update to that tile first.
    // Measured: n = 256 0.141 -> 0.128 ms, n = 512 0.273 -> 0.247 ms.  With
    // more rest tiles the extra product in phase 1 costs more than the
    // overlap gains (n = 768: 0.43 against 0.39-0.41 ms; n = 2048: 2.27
    // against 2.20 ms).
    const bool merged = m.fb == bs::FB_SMALL && rest_tiles * m.batch < 0.5 * m.sms;
    for (int K = 0; merged && K + 1 < nb && e == cudaSuccess; ++K) {
        // s: phase 3 of round K but tile (K+1,K+1), after phase 2 of round K
        if (forked) e = cudaStreamWaitEvent(s, c.side_done, 0);
        forked = false;
        if (e == cudaSuccess) e = bs::launch_phase3(is_int, m, K, bs::P3_ALL_OFF, s);
        if (e == cudaSuccess) e = cudaEventRecord(c.main_done[K & 1], s);
        // side: phase 1 of round K+1 after phase 3 of round K-1, phase 2 of
        // round K+1 after phase 3 of round K
        if (e == cudaSuccess) e = cudaStreamWaitEvent(c.side, c.main_done[(K + 1) & 1], 0);
        if (e != cudaSuccess) break;
        forked = true;
        e = bs::launch_phase1(is_int, m, K + 1, true, c.side);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(c.side, c.main_done[K & 1], 0);
        if (e == cudaSuccess) e = bs::launch_phase2(is_int, m, K + 1, c.side);
        cudaError_t r = cudaEventRecord(c.side_done, c.side);
        if (e == cudaSuccess) e = r;
    }
    for (int K = 0; !merged && K + 1 < nb && e == cudaSuccess; ++K) {
        if (!tight) {
            // REST(K) after phase 2 of round K
            e = rest(K, forked ? c.side_done : nullptr);
            forked = false;
            if (e != cudaSuccess) break;
        }
        // side: after REST(K-1), NEXT(K) then phases 1 and 2 of round K+1
        e = cudaStreamWaitEvent(c.side, c.main_done[(K + 1) & 1], 0);
        if (e != cudaSuccess) break;
        forked = true;
        e = bs::launch_phase3(is_int, m, K, bs::P3_NEXT, c.side);
        if (e == cudaSuccess && tight) e = cudaEventRecord(c.next_done, c.side);
        if (e == cudaSuccess) e = bs::launch_phase1(is_int, m, K + 1, false, c.side);
        if (e == cudaSuccess) e = bs::launch_phase2(is_int, m, K + 1, c.side);
        cudaError_t r = cudaEventRecord(c.side_done, c.side);
        if (e == cudaSuccess) e = r;
        if (e == cudaSuccess && tight) e = rest(K, c.next_done);
    }
    // always join the side stream back, on success or failure
    if (forked) {
        cudaError_t j = cudaStreamWaitEvent(s, c.side_done, 0);
        if (e == cudaSuccess) e = j;
    }
    if (e == cudaSuccess) e = bs::launch_phase3(is_int, m, nb - 1, bs::P3_ALL, s);
    if (e == cudaSuccess && m.sym) e = bs::launch_mirror(is_int, m, s);
    release_side(d, c);
    return e;
}

bs_status cuda_status(cudaError_t e) { return e == cudaSuccess ? BS_OK : BS_ERR_CUDA; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Common argument checks.  Returns BS_OK and fills `m`, or an error.
bs_status check_args(const void* U, const void* L, bool bounds, int n, int ld,
                     long long bstride, int batch, int mode, bs::Mats* m) {
    const int known = BS_DTYPE_MASK | BS_PERK | BS_RULE_LITERAL | BS_VALIDATE | BS_TILE_64 |
                      BS_TILE_128 | BS_NO_LOOKAHEAD | BS_SYMMETRIC | BS_PERK_PAIRED |
                      BS_ONE_LAUNCH | BS_PAIRED_ROUNDS;
    if (mode & ~known) return BS_ERR_ARG;
    if ((mode & BS_TILE_64) && (mode & BS_TILE_128)) return BS_ERR_ARG;
    if ((mode & BS_PERK_PAIRED) && !(mode & BS_PERK)) return BS_ERR_ARG;
    if ((mode & BS_ONE_LAUNCH) && (mode & (BS_PERK | BS_TILE_128 | BS_NO_LOOKAHEAD)))
        return BS_ERR_ARG;
    if ((mode & BS_PAIRED_ROUNDS) && (mode & (BS_PERK | BS_ONE_LAUNCH | BS_NO_LOOKAHEAD)))
        return BS_ERR_ARG;
    if ((mode & BS_DTYPE_MASK) > BS_INT32_Q10) return BS_ERR_ARG;
    if (n < 0 || batch < 0) return BS_ERR_ARG;
    if (n > 0 && ld < n) return BS_ERR_ARG;
    if (n > 0 && batch > 0) {
        if (!U || (bounds && !L)) return BS_ERR_ARG;
        if (bounds && U == L) return BS_ERR_ARG;
        const long long span = (long long)(n - 1) * ld + n;
        if (batch > 1 && bstride < span) return BS_ERR_ARG;
        if (!aligned(U, 4) || (bounds && !aligned(L, 4))) return BS_ERR_ALIGN;
    }
    m->U = const_cast<void*>(U);
    m->L = bounds ? const_cast<void*>(L) : nullptr;
    m->n = n;
    m->ld = ld;
    m->bstride = batch > 1 ? bstride : 0;
    m->batch = batch;
    m->vec = (ld % 4 == 0) && aligned(U, 16) && (!bounds || aligned(L, 16)) &&
             (batch <= 1 || bstride % 4 == 0);
    m->fb = (mode & BS_ONE_LAUNCH) ? bs::FB_SMALL : choose_tile(n, batch, mode, bounds);
    m->sym = (mode & BS_SYMMETRIC) != 0;
    m->sms = 1;
    return BS_OK;
}

bs_status validate(const bs::Mats& m, bool is_int, cudaStream_t s) {
    unsigned long long* scr = nullptr;
    cudaError_t e = device_scratch(&scr);
    if (e != cudaSuccess) return BS_ERR_CUDA;
    unsigned int* flags = reinterpret_cast<unsigned int*>(scr + 1);
    e = cudaMemsetAsync(flags, 0, sizeof(unsigned int), s);
    if (e == cudaSuccess) e = bs::launch_validate(is_int, m, flags, s);
    unsigned int h = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h, flags, sizeof h, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return BS_ERR_CUDA;
    if (h & (bs::VF_DIAG | bs::VF_NEG | bs::VF_NAN | bs::VF_LINF | bs::VF_ASYM)) return BS_ERR_INPUT;
    if (h & bs::VF_RANGE) return BS_ERR_RANGE;
    return BS_OK;
}

bs_status smooth(void* U, void* L, bool bounds, int n, int ld, long long bstride, int batch,
                 cudaStream_t s, int mode) {
    bs::Mats m;
    bs_status st = check_args(U, L, bounds, n, ld, bstride, batch, mode, &m);
    if (st != BS_OK) return st;
    const bool perk = (mode & BS_PERK) != 0;
    const bool literal = bounds && (mode & BS_RULE_LITERAL) != 0;
    if (literal && !perk) return BS_ERR_ARG;
    if (perk && (mode & BS_SYMMETRIC)) return BS_ERR_ARG;
    if (n == 0 || batch == 0) return BS_OK;
    const bool is_int = (mode & BS_DTYPE_MASK) == BS_INT32_Q10;
    DeviceState* d = nullptr;
    if (device_state(&d) != cudaSuccess) return BS_ERR_CUDA;
    m.sms = d->sms;
    if (mode & BS_VALIDATE) {
        st = validate(m, is_int, s);
        if (st != BS_OK) return st;
    }
    cudaError_t e = cudaSuccess;
    if (perk) {
        // plain: every round alone, then its row and column (perk.cu);
        // paired: two rounds per pass, each pass followed by its rows and
        // columns, and with n odd the last round in the plain form
        int k = 0;
        if (mode & BS_PERK_PAIRED)
            for (; k + 1 < n && e == cudaSuccess; k += 2)
                e = bs::launch_round2(is_int, m, k, literal, s);
        for (; k < n && e == cudaSuccess; ++k) {
            e = bs::launch_round(is_int, m, k, literal, s);
            if (e == cudaSuccess && bounds) e = bs::launch_cross(is_int, m, k, s);
        }
    } else if (mode & BS_ONE_LAUNCH) {
        e = bs::launch_fused(is_int, m, s);
    } else {
        e = run_blocked(is_int, m, s, (mode & BS_NO_LOOKAHEAD) == 0,
                        (mode & BS_PAIRED_ROUNDS) != 0, d);
    }
    return cuda_status(e);
}

}  // namespace

// ---- launch bookkeeping used by the kernel translation units ---------------

namespace bs {

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void before_launch(cudaStream_t s, int) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    t_pending = nullptr;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on) return;
    if (g_prof.size() >= kMaxProf) {
        g_prof_overflow = true;
        return;
    }
    cudaEvent_t a;
    if (cudaEventCreate(&a) != cudaSuccess) return;
    cudaEventRecord(a, s);
    t_pending = a;
}

void after_launch(cudaStream_t s, int phase) {
    if (!t_pending) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    cudaEvent_t b;
    if (cudaEventCreate(&b) != cudaSuccess) {
        cudaEventDestroy(t_pending);
        t_pending = nullptr;
        return;
    }
    cudaEventRecord(b, s);
    g_prof.push_back(ProfRec{t_pending, b, phase});
    t_pending = nullptr;
}

}  // namespace bs

// ---- the C ABI -------------------------------------------------------------

extern "C" {

bs_status bs_smooth_upper(void* U, int n, int ld, bs_stream_t stream, int mode) {
    // rule bits have no meaning for the upper bound alone
    return smooth(U, nullptr, false, n, ld, 0, 1, stream, mode & ~BS_RULE_LITERAL);
}

bs_status bs_smooth_bounds(void* U, void* L, int n, int ld, bs_stream_t stream, int mode) {
    return smooth(U, L, true, n, ld, 0, 1, stream, mode);
}

bs_status bs_smooth_bounds_batched(void* U, void* L, int n, int ld, long long batch_stride,
                                   int batch, bs_stream_t stream, int mode) {
    return smooth(U, L, true, n, ld, batch_stride, batch, stream, mode);
}

bs_status bs_check_feasible(const void* U, const void* L, int n, int ld, bs_stream_t stream,
                            int mode, long long* out_count, unsigned char* mask) {
    if (!out_count) return BS_ERR_ARG;
    bs::Mats m;
    bs_status st = check_args(U, L, true, n, ld, 0, 1, mode & BS_DTYPE_MASK, &m);
    if (st != BS_OK) return st;
    if (n == 0) {
        *out_count = 0;
        return BS_OK;
    }
    const bool is_int = (mode & BS_DTYPE_MASK) == BS_INT32_Q10;
    unsigned long long* scr = nullptr;
    cudaError_t e = device_scratch(&scr);
    if (e == cudaSuccess) e = cudaMemsetAsync(scr, 0, sizeof(unsigned long long), stream);
    if (e == cudaSuccess) e = bs::launch_feasible(is_int, m, mask, scr, stream);
    unsigned long long h = 0;
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&h, scr, sizeof h, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return BS_ERR_CUDA;
    *out_count = (long long)h;
    return BS_OK;
}

const char* bs_strerror(bs_status status) {
    switch (status) {
        case BS_OK: return "success";
        case BS_ERR_ARG: return "invalid argument (n, ld, batch, stride, pointer or mode bits)";
        case BS_ERR_ALIGN: return "matrix pointer not aligned to its element size";
        case BS_ERR_RANGE: return "int32 bound outside [0, 2^30)";
        case BS_ERR_CUDA: return "CUDA launch or call failed";
        case BS_ERR_TIMEOUT: return "bounded device wait ran out";
        case BS_ERR_INPUT: return "input violates preconditions (diagonal, sign, NaN, infinite lower bound)";
    }
    return "unknown status";
}

long long bs_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int bs_one_launch_cluster(void) { return bs::fused_cluster_size(); }

bs_status bs_schedule_info(int n, int batch, int mode, int bounds, int* tile, int* pairs) {
    if (!tile || !pairs) return BS_ERR_ARG;
    // the argument rules of a smoothing call on a contiguous layout; the two
    // addresses are placeholders that check_args never dereferences
    const int ld = n > 0 ? n : 1;
    const long long span = n > 0 ? (long long)(n - 1) * ld + n : 1;
    bs::Mats m;
    bs_status st = check_args(reinterpret_cast<const void*>(256), reinterpret_cast<const void*>(512),
                              bounds != 0, n, ld, span, batch, mode, &m);
    if (st != BS_OK) return st;
    const bool perk = (mode & BS_PERK) != 0;
    if ((bounds && (mode & BS_RULE_LITERAL) && !perk) || (perk && (mode & BS_SYMMETRIC)))
        return BS_ERR_ARG;
    const int nb = n > 0 ? (n + m.fb - 1) / m.fb : 0;
    *tile = perk ? 0 : m.fb;
    // run_blocked: look-ahead from three block rows, then the pair rule
    *pairs = !perk && !(mode & BS_ONE_LAUNCH) && !(mode & BS_NO_LOOKAHEAD) && nb >= 3 &&
             ((mode & BS_PAIRED_ROUNDS) || pairs_pay(m, nb));
    return BS_OK;
}

bs_status bs_profile_begin(void) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (auto& r : g_prof) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g_prof.clear();
    g_prof_overflow = false;
    g_prof_on = true;
    return BS_OK;
}

bs_status bs_profile_end(bs_profile* out) {
    std::vector<ProfRec> recs;
    bool overflow;
    {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        g_prof_on = false;
        recs.swap(g_prof);
        overflow = g_prof_overflow;
    }
    bs_profile p{};
    cudaError_t first = cudaSuccess;
    for (auto& r : recs) {
        float ms = 0.f;
        cudaError_t e = cudaEventSynchronize(r.b);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.a, r.b);
        if (e == cudaSuccess && r.phase >= 0 && r.phase < BS_PROFILE_PHASES) {
            p.ms[r.phase] += ms;
            p.launches[r.phase] += 1;
        } else if (first == cudaSuccess) {
            first = e;
        }
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    p.overflow = overflow ? 1 : 0;
    if (out) *out = p;
    return cuda_status(first);
}

}  // extern "C"
