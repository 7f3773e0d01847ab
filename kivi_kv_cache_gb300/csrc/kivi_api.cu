// kivi_api.cu -- the extern "C" boundary of libkivi_gb300.so (declared in
// include/kivi.h). Every entry point validates its arguments on the host,
// returns a status without launching when a check fails, and otherwise
// launches the CUDA kernels on the caller's stream. No allocation, no state
// beyond a per-device cache of the SM count.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "../../include/kivi.h"
#include "kivi_launch.h"

using namespace kivi;

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
}  // namespace

int kivi::sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 152;  // GB300; only used for sizing when no device is visible
    }
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            return 152;
        }
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The `bits` argument of every entry point: the bit width, optionally ORed
// with KIVI_SCALE_F16 (scales stored as fp16). Any other high bit leaves a
// width outside {2, 4}, which the shape check refuses.
bool scale_f16_of(int bits) { return (bits & KIVI_SCALE_F16) != 0; }
int width_of(int bits) { return bits & ~KIVI_SCALE_F16; }
// The decode's `bits` may also carry KIVI_DECODE_STORE_READY (the store is
// not written by the kernel that precedes the call on its stream).
bool store_ready_of(int bits) { return (bits & KIVI_DECODE_STORE_READY) != 0; }
int decode_bits(int bits) { return bits & ~KIVI_DECODE_STORE_READY; }

bool head_dim_ok(int D) { return D == 64 || D == 128 || D == 256; }

// Every op: D in {64, 128, 256}, G in {32, 64, 128} with G <= D (a value
// group lies within one token row), 2 or 4 bits.
kivi_status shape_check(int D, int G, int bits) {
    if (!head_dim_ok(D) || (G != 32 && G != 64 && G != 128) || G > D || (bits != 2 && bits != 4))
        return KIVI_ERR_UNSUPPORTED;
    return KIVI_OK;
}

kivi_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KIVI_OK : KIVI_ERR_CUDA; }

// Split plan for the decode, run by the one-warp-per-tile kernel: each warp of
// a CTA takes a run of tiles_per_warp tiles (32-token store tiles, then
// 16-token residual tiles), sized for about kMmaWarpsPerSm warps per SM over
// the whole batch. CTAs have 4 warps, or 8 when 4-warp CTAs would leave a
// head group more than kMmaMaxSplits4 partials to merge. Groups of 1, 2 or 4
// query heads per KV head run as one head group; any other group size runs in
// q_sub = ceil(gq / 4) sub-groups of up to 4 heads, each a head group of its
// own (the sub-groups of one split read the same tiles side by side, so L2
// serves the repeated reads). When the batch has more head groups than the
// workspace has merge counters, each gets one split.
#ifndef KIVI_DECODE_MMA_WARPS_PER_SM
#define KIVI_DECODE_MMA_WARPS_PER_SM 24
#endif
#ifndef KIVI_DECODE_MMA_MAX_SPLITS4
#define KIVI_DECODE_MMA_MAX_SPLITS4 16
#endif
// Warp-pair kernel: 0 never, 1 always, 2 when the one-warp-per-tile plan gives
// warps at most kPairMaxWarpTiles tiles and the pair plan at most
// kPairMaxSplits splits per head (small batches with short caches, where one
// tile's chain and the merge bound the launch). A pair takes at least
// kPairMinTiles tiles.
#ifndef KIVI_DECODE_PAIR_MODE
#define KIVI_DECODE_PAIR_MODE 2
#endif
#ifndef KIVI_DECODE_PAIR_MAX_WARP_TILES
#define KIVI_DECODE_PAIR_MAX_WARP_TILES 1
#endif
#ifndef KIVI_DECODE_PAIR_MAX_SPLITS
#define KIVI_DECODE_PAIR_MAX_SPLITS 24
#endif
#ifndef KIVI_DECODE_PAIR_MIN_TILES
#define KIVI_DECODE_PAIR_MIN_TILES 1
#endif
#ifndef KIVI_DECODE_PAIRS_PER_SM
#define KIVI_DECODE_PAIRS_PER_SM 8
#endif
constexpr int kPairMode = KIVI_DECODE_PAIR_MODE;
constexpr int kPairMaxWarpTiles = KIVI_DECODE_PAIR_MAX_WARP_TILES;
constexpr int kPairMinTiles = KIVI_DECODE_PAIR_MIN_TILES;
constexpr int kPairMaxSplits = KIVI_DECODE_PAIR_MAX_SPLITS;
constexpr int kPairsPerSm = KIVI_DECODE_PAIRS_PER_SM;
constexpr int kMmaWarpsPerSm = KIVI_DECODE_MMA_WARPS_PER_SM;
#ifndef KIVI_DECODE_MMA_WARPS_PER_SM_2BIT
#define KIVI_DECODE_MMA_WARPS_PER_SM_2BIT 16
#endif
constexpr int kMmaWarpsPerSm2 = KIVI_DECODE_MMA_WARPS_PER_SM_2BIT;
constexpr int kMmaMaxSplits4 = KIVI_DECODE_MMA_MAX_SPLITS4;
#ifndef KIVI_DECODE_ONE_WAVE
#define KIVI_DECODE_ONE_WAVE 1
#endif
constexpr bool kOneWave = KIVI_DECODE_ONE_WAVE != 0;
#ifndef KIVI_DECODE_BALANCE
#define KIVI_DECODE_BALANCE 1
#endif
constexpr bool kBalance = KIVI_DECODE_BALANCE != 0;
#ifndef KIVI_DECODE_SHORT_RUNS
#define KIVI_DECODE_SHORT_RUNS 1
#endif
constexpr bool kShortRuns = KIVI_DECODE_SHORT_RUNS != 0;
constexpr long long kShortRunTiles = 8;       // longest warp run the 2-warp plan serves
constexpr long long kShortRunMaxSplits = 24;  // most splits per head group it takes

bool mma_group(int gq) { return gq == 1 || gq == 2 || gq == 4; }

// pair_ok: the warp-pair kernel may run (it reads stores of group size 32 at
// head dim 128 only). D: head dim; D = 256 keeps 8 warps per SM resident
// instead of 16.
DecodePlan make_plan(int B, int Hkv, int Hq, int S_q, int n_res, int bits, bool pair_ok, int D) {
    DecodePlan p;
    const int gq = Hkv > 0 && Hq >= Hkv ? Hq / Hkv : 1;
    p.q_sub = mma_group(gq) ? 1 : (gq + 3) / 4;
    p.n_store_tiles = (S_q + kG - 1) / kG;
    p.n_tiles = p.n_store_tiles + (n_res + kResTileTokensMma - 1) / kResTileTokensMma;
    const long long heads = (long long)B * Hkv * p.q_sub;  // head groups (batch, KV head, sub-group)
    // 2-bit tiles carry half the codes: fewer, longer-running warps measured faster
    const long long target = (long long)(bits == 2 ? kMmaWarpsPerSm2 : kMmaWarpsPerSm) * sm_count();
    long long tpw = (heads * p.n_tiles + target - 1) / target;
    if (tpw < 1) tpw = 1;
    p.warps_per_cta = (p.n_tiles + 4 * tpw - 1) / (4 * tpw) > kMmaMaxSplits4 ? 8 : 4;
    if (heads > kMergeCounters) tpw = (p.n_tiles + p.warps_per_cta - 1) / p.warps_per_cta;  // one split each
    if (kOneWave && tpw >= 2 && heads <= kMergeCounters) {
        // a grid of multi-tile warps that just spills into a second wave of
        // resident CTAs (at most 1.25 waves) takes up to half again as many
        // tiles per warp instead
        const long long slots = (long long)((D == 256 ? 8 : 16) / p.warps_per_cta) * sm_count();  // resident CTAs
        auto ctas = [&](long long t) { return heads * ((p.n_tiles + p.warps_per_cta * t - 1) / (p.warps_per_cta * t)); };
        if (ctas(tpw) > slots && 4 * ctas(tpw) <= 5 * slots) {
            long long t = tpw;
            while (ctas(t) > slots && 2 * t < 3 * tpw + 2) ++t;
            if (ctas(t) <= slots) tpw = t;
        }
    }
    p.tiles_per_warp = (int)tpw;
    p.tiles_per_split = (int)(p.warps_per_cta * tpw);
    p.pair_kernel = 0;
    if (pair_ok && mma_group(gq) && (kPairMode == 1 || (kPairMode == 2 && tpw <= kPairMaxWarpTiles && heads <= kMergeCounters))) {
        const long long slots = (long long)kPairsPerSm * sm_count();
        long long tpp = (heads * p.n_tiles + slots - 1) / slots;  // tiles per pair
        if (tpp < kPairMinTiles) tpp = kPairMinTiles;
        if (heads > kMergeCounters) tpp = (p.n_tiles + kPairsPerCta - 1) / kPairsPerCta;
        const long long splits = (p.n_tiles + kPairsPerCta * tpp - 1) / (kPairsPerCta * tpp);
        if (kPairMode == 1 || splits <= kPairMaxSplits) {
            p.pair_kernel = 1;
            p.tiles_per_warp = (int)tpp;
            p.tiles_per_split = (int)(kPairsPerCta * tpp);
        }
    }
    p.n_split = (p.n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    if (kBalance && heads <= kMergeCounters) {
        // A one-warp-per-tile grid of more than one CTA per SM but less than
        // one wave leaves some SMs one CTA more than others, and those set the
        // pace. When more splits fill every SM's resident slots (at least 95 %
        // of them), take them: each split gets fewer tiles and every SM the
        // same load. Plans that merge inside a cluster (at most 16 splits)
        // keep that merge.
        const long long S = sm_count();
        const long long cps = p.pair_kernel ? 16 / (2 * kPairsPerCta) : (D == 256 ? 8 : 16) / p.warps_per_cta;
        const long long ctas = heads * p.n_split;
        const int wpc = p.pair_kernel ? kPairsPerCta : p.warps_per_cta;  // warps (pairs) sharing a split
        if (ctas > cps * S && 3 * ctas <= 4 * cps * S && p.n_split > 1) {
            // a grid that spills just past one wave (at most 4/3 of a wave: the
            // multi-tile rule above did not apply) takes fewer splits and
            // stays in one wave; its warps take a tile or so more each
            const long long n2 = cps * S / heads;
            if (n2 >= 1) {
                p.n_split = (int)n2;
                p.tiles_per_split = (p.n_tiles + p.n_split - 1) / p.n_split;
                p.tiles_per_warp = (p.tiles_per_split + wpc - 1) / wpc;
            }
        } else if (!p.pair_kernel && ctas > S && ctas < cps * S) {
            long long n2 = cps * S / heads;
            if (n2 > p.n_tiles) n2 = p.n_tiles;
            const bool keeps_cluster = p.n_split <= kMaxClusterSplits && n2 > kMaxClusterSplits;
            if (n2 > p.n_split && !keeps_cluster && 20 * heads * n2 >= 19 * cps * S) {
                p.n_split = (int)n2;
                p.tiles_per_split = (p.n_tiles + p.n_split - 1) / p.n_split;
                p.tiles_per_warp = (p.tiles_per_split + p.warps_per_cta - 1) / p.warps_per_cta;
            }
        }
    }
    if (kShortRuns && !p.pair_kernel && heads <= kMergeCounters && D == 128) {
        // Short warp runs on a grid of 4- or 8-warp CTAs that spills past
        // one wave, or that leaves each warp a third more tiles than a finer
        // split would: 2-warp CTAs (8 per SM) fill one wave with more splits
        // per head group, so its warps' runs are shorter (B=16 x 3072 tokens:
        // 27.1 -> 24.6 us). At equal or nearly equal runs the extra partials
        // and CTA merges cost more than they save, so the plan stays; so do
        // plans that would need more than 24 splits per head group, whose
        // merges read too many partials (B=1 x 65536: 147 splits of 2 warps
        // took 37.4 us against 31.2 us).
        const long long S = sm_count();
        const long long slots = (long long)(16 / p.warps_per_cta) * S;
        const long long ctas = heads * p.n_split;
        const long long tpw = (p.tiles_per_split + p.warps_per_cta - 1) / p.warps_per_cta;
        const long long run = ((ctas + slots - 1) / slots) * tpw;  // tiles a warp slot runs
        long long n2 = 8 * S / heads;
        if (n2 > p.n_tiles) n2 = p.n_tiles;
        if (n2 > kShortRunMaxSplits) n2 = kShortRunMaxSplits;
        if (n2 >= 1) {
            const long long tps2 = (p.n_tiles + n2 - 1) / n2;
            const long long run2 = (tps2 + 1) / 2;
            if (run2 <= kShortRunTiles && (ctas > slots ? run2 < run : 3 * run2 <= 2 * run)) {
                p.warps_per_cta = 2;
                p.n_split = (int)((p.n_tiles + tps2 - 1) / tps2);
                p.tiles_per_split = (int)tps2;
                p.tiles_per_warp = (int)run2;
            }
        }
    }
    return p;
}

// Workspace: [merge counters, KIVI_DECODE_COUNTER_BYTES][part_o, 256-aligned][part_ml]
size_t part_o_bytes(int B, int Hq, int D, const DecodePlan& p) {
    return (((size_t)B * Hq * p.n_split * D * sizeof(float)) + 255) & ~(size_t)255;
}

size_t workspace_bytes(int B, int Hq, int D, const DecodePlan& p) {
    if (p.n_split <= 1) return 0;
    const size_t ml = (size_t)B * Hq * p.n_split * 2 * sizeof(float);
    return (size_t)KIVI_DECODE_COUNTER_BYTES + part_o_bytes(B, Hq, D, p) + ml;
}

kivi_status flush_check(const void* x, int BH, int S, int x_bh_stride, int D, int G, int bits,
                        int R, const void* codes, const void* scale, const void* zero,
                        int s_off, int s_cap, bool keys, int* n_flush) {
    kivi_status st = shape_check(D, G, bits);
    if (st != KIVI_OK) return st;
    if (BH <= 0 || S < 0 || x_bh_stride < S || R < 0 || s_cap <= 0 || s_cap % G != 0 || s_off < 0)
        return KIVI_ERR_INVALID_ARG;
    if (keys && s_off % G != 0) return KIVI_ERR_INVALID_ARG;
    const int n = kivi_flush_count(S, R, G);
    if (n < 0 || (long long)s_off + n > s_cap) return KIVI_ERR_INVALID_ARG;
    if (n > 0 && (!x || !codes || !scale || !zero)) return KIVI_ERR_INVALID_ARG;
    if (n > 0 && (!aligned16(x) || !aligned16(codes) || !aligned16(scale) || !aligned16(zero)))
        return KIVI_ERR_ALIGNMENT;
    *n_flush = n;
    return KIVI_OK;
}

FlushArgs flush_args(const void* x, int BH, int x_bh_stride, int n, void* codes, float* scale,
                     void* zero, int s_off, int s_cap, int G, int D, bool hs) {
    FlushArgs a;
    a.G = G;
    a.D = D;
    a.scale_f16 = hs;
    a.x = static_cast<const __half*>(x);
    a.x_bh_stride = x_bh_stride;
    a.BH = BH;
    a.n_flush = n;
    a.codes = static_cast<uint8_t*>(codes);
    a.scale = scale;
    a.zero = static_cast<__half*>(zero);
    a.s_off = s_off;
    a.s_cap = s_cap;
    return a;
}

kivi_status flush_one(int axis, const void* x, int BH, int S, int x_bh_stride, int D, int G,
                      int bits, int R, void* codes, float* scale, void* zero, int s_off,
                      int s_cap, int* n_flushed, kivi_stream_t stream) {
    const bool hs = scale_f16_of(bits);
    bits = width_of(bits);
    int n = 0;
    kivi_status st = flush_check(x, BH, S, x_bh_stride, D, G, bits, R, codes, scale, zero, s_off,
                                 s_cap, axis == 0, &n);
    if (st != KIVI_OK) return st;
    if (n_flushed) *n_flushed = n;
    if (n == 0) return KIVI_OK;
    return from_cuda(launch_flush(axis, flush_args(x, BH, x_bh_stride, n, codes, scale, zero, s_off, s_cap, G, D, hs),
                                  bits, reinterpret_cast<cudaStream_t>(stream)));
}

// Fake quantization of keys (do_k) and/or values (do_v): the first
// kivi_flush_count(S, R, G) tokens of each input become their KIVI
// reconstructions in the output; the remaining tokens are copied unchanged
// unless the output is the input (in place).
kivi_status fake_quant(const void* k, const void* v, bool do_k, bool do_v, int BH, int S, int x_bh_stride,
                       int D, int G, int bits, int R, void* k_out, void* v_out, int out_bh_stride,
                       int* n_quantized, kivi_stream_t stream) {
    const bool hs = scale_f16_of(bits);
    bits = width_of(bits);
    kivi_status st = shape_check(D, G, bits);
    if (st != KIVI_OK) return st;
    if (BH <= 0 || S < 0 || R < 0 || x_bh_stride < S || out_bh_stride < S) return KIVI_ERR_INVALID_ARG;
    const int n = kivi_flush_count(S, R, G);
    if (n < 0) return KIVI_ERR_INVALID_ARG;
    if (n_quantized) *n_quantized = n;
    if (S == 0) return KIVI_OK;
    if ((do_k && (!k || !k_out)) || (do_v && (!v || !v_out))) return KIVI_ERR_INVALID_ARG;
    // the output either is the input (same place and stride) or leaves it alone
    if ((do_k && k_out == k && out_bh_stride != x_bh_stride) || (do_v && v_out == v && out_bh_stride != x_bh_stride))
        return KIVI_ERR_INVALID_ARG;
    if ((do_k && (!aligned16(k) || !aligned16(k_out))) || (do_v && (!aligned16(v) || !aligned16(v_out))))
        return KIVI_ERR_ALIGNMENT;
    const cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);
    if (n > 0) {
        FlushArgs ka = flush_args(do_k ? k : v, BH, x_bh_stride, n, nullptr, nullptr, nullptr, 0, G, G, D, hs);
        FlushArgs va = flush_args(do_v ? v : k, BH, x_bh_stride, n, nullptr, nullptr, nullptr, 0, G, G, D, hs);
        ka.fq = static_cast<__half*>(do_k ? k_out : v_out);
        va.fq = static_cast<__half*>(do_v ? v_out : k_out);
        ka.fq_bh_stride = va.fq_bh_stride = out_bh_stride;
        cudaError_t e = launch_fake_quant(ka, va, do_k, do_v, bits, strm);
        if (e != cudaSuccess) return from_cuda(e);
    }
    // tokens [n, S) stay fp16: copy them behind the reconstructions
    const int tail = S - n;
    const bool copy_k = do_k && k_out != k, copy_v = do_v && v_out != v;
    if (tail > 0 && (copy_k || copy_v)) {
        const __half* src0 = static_cast<const __half*>(copy_k ? k : v) + (long long)n * D;
        const __half* src1 = copy_k && copy_v ? static_cast<const __half*>(v) + (long long)n * D : nullptr;
        __half* dst0 = static_cast<__half*>(copy_k ? k_out : v_out);
        __half* dst1 = copy_k && copy_v ? static_cast<__half*>(v_out) : nullptr;
        return from_cuda(
            launch_residual_append(src0, src1, x_bh_stride, tail, dst0, dst1, BH, out_bh_stride, n, D, strm));
    }
    return KIVI_OK;
}

}  // namespace

// KIVI_OK, or KIVI_ERR_UNSUPPORTED for a head dim, group size or bit width
// (bits may carry KIVI_SCALE_F16) outside the compiled set.
int kivi::shape_status(int D, int group_size, int bits) {
    return (int)shape_check(D, group_size, width_of(bits));
}

// Workspace bytes of the plan kivi_decode_attend takes for exactly these
// arguments (bits may carry KIVI_SCALE_F16); 0 for a single-split plan or
// for arguments the decode rejects.
size_t kivi::decode_workspace_need(int B, int Hq, int Hkv, int S_q, int n_res, int D, int group_size, int bits) {
    bits = decode_bits(bits);
    const bool hs = scale_f16_of(bits);
    bits = width_of(bits);
    if (shape_check(D, group_size, bits) != KIVI_OK || B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 ||
        Hq / Hkv > 64 || S_q < 0 || n_res < 0 || S_q + n_res == 0)
        return 0;
    return workspace_bytes(B, Hq, D, make_plan(B, Hkv, Hq, S_q, n_res, bits, group_size == kG && D == kD && !hs, D));
}

extern "C" {

kivi_status kivi_fake_quant_keys(const void* x_f16, int BH, int S, int x_bh_stride, int D, int group_size,
                                 int bits, int residual_length, void* out_f16, int out_bh_stride,
                                 int* n_quantized, kivi_stream_t stream) {
    return fake_quant(x_f16, nullptr, true, false, BH, S, x_bh_stride, D, group_size, bits, residual_length,
                      out_f16, nullptr, out_bh_stride, n_quantized, stream);
}

kivi_status kivi_fake_quant_values(const void* x_f16, int BH, int S, int x_bh_stride, int D, int group_size,
                                   int bits, int residual_length, void* out_f16, int out_bh_stride,
                                   int* n_quantized, kivi_stream_t stream) {
    return fake_quant(nullptr, x_f16, false, true, BH, S, x_bh_stride, D, group_size, bits, residual_length,
                      nullptr, out_f16, out_bh_stride, n_quantized, stream);
}

kivi_status kivi_fake_quant_kv(const void* k_f16, const void* v_f16, int BH, int S, int x_bh_stride, int D,
                               int group_size, int bits, int residual_length, void* k_out_f16,
                               void* v_out_f16, int out_bh_stride, int* n_quantized, kivi_stream_t stream) {
    return fake_quant(k_f16, v_f16, true, true, BH, S, x_bh_stride, D, group_size, bits, residual_length,
                      k_out_f16, v_out_f16, out_bh_stride, n_quantized, stream);
}

const char* kivi_status_string(kivi_status s) {
    switch (s) {
        case KIVI_OK: return "KIVI_OK";
        case KIVI_ERR_INVALID_ARG: return "KIVI_ERR_INVALID_ARG";
        case KIVI_ERR_UNSUPPORTED: return "KIVI_ERR_UNSUPPORTED";
        case KIVI_ERR_WORKSPACE: return "KIVI_ERR_WORKSPACE";
        case KIVI_ERR_CUDA: return "KIVI_ERR_CUDA";
        case KIVI_ERR_ALIGNMENT: return "KIVI_ERR_ALIGNMENT";
    }
    return "KIVI_ERR_UNKNOWN";
}

int kivi_version(void) { return 100; }

kivi_status kivi_wait_timeouts(unsigned int* count, int reset) {
    if (count == nullptr) return KIVI_ERR_INVALID_ARG;
    return from_cuda(kivi::read_wait_timeouts(count, reset != 0));
}

int kivi_flush_count(int n_res, int residual_length, int group_size) {
    if (n_res < 0 || residual_length < 0 || group_size <= 0) return -1;
    if (n_res == 0) return 0;
    if (residual_length == 0) return n_res;
    const int over = n_res - residual_length;
    if (over < group_size) return 0;
    return (over / group_size) * group_size;
}

kivi_status kivi_flush_keys(const void* x_f16, int BH, int S, int x_bh_stride, int D,
                            int group_size, int bits, int residual_length, void* codes_u8,
                            float* scale, void* zero_f16, int s_off, int s_cap, int* n_flushed,
                            kivi_stream_t stream) {
    return flush_one(0, x_f16, BH, S, x_bh_stride, D, group_size, bits, residual_length, codes_u8,
                     scale, zero_f16, s_off, s_cap, n_flushed, stream);
}

kivi_status kivi_flush_values(const void* x_f16, int BH, int S, int x_bh_stride, int D,
                              int group_size, int bits, int residual_length, void* codes_u8,
                              float* scale, void* zero_f16, int s_off, int s_cap, int* n_flushed,
                              kivi_stream_t stream) {
    return flush_one(1, x_f16, BH, S, x_bh_stride, D, group_size, bits, residual_length, codes_u8,
                     scale, zero_f16, s_off, s_cap, n_flushed, stream);
}

kivi_status kivi_flush_kv(const void* k_f16, const void* v_f16, int BH, int S, int x_bh_stride,
                          int D, int group_size, int bits, int residual_length, void* kcodes_u8,
                          float* kscale, void* kzero_f16, void* vcodes_u8, float* vscale,
                          void* vzero_f16, int s_off, int s_cap, int* n_flushed,
                          kivi_stream_t stream) {
    const bool hs = scale_f16_of(bits);
    bits = width_of(bits);
    int nk = 0, nv = 0;
    kivi_status st = flush_check(k_f16, BH, S, x_bh_stride, D, group_size, bits, residual_length,
                                 kcodes_u8, kscale, kzero_f16, s_off, s_cap, true, &nk);
    if (st != KIVI_OK) return st;
    st = flush_check(v_f16, BH, S, x_bh_stride, D, group_size, bits, residual_length, vcodes_u8,
                     vscale, vzero_f16, s_off, s_cap, false, &nv);
    if (st != KIVI_OK) return st;
    if (n_flushed) *n_flushed = nk;
    if (nk == 0) return KIVI_OK;
    return from_cuda(launch_flush_kv(
        flush_args(k_f16, BH, x_bh_stride, nk, kcodes_u8, kscale, kzero_f16, s_off, s_cap, group_size, D, hs),
        flush_args(v_f16, BH, x_bh_stride, nv, vcodes_u8, vscale, vzero_f16, s_off, s_cap, group_size, D, hs), bits,
        reinterpret_cast<cudaStream_t>(stream)));
}

kivi_status kivi_dequant(kivi_axis axis, const void* codes_u8, const float* scale,
                         const void* zero_f16, int BH, int S, int D, int group_size, int bits,
                         int s_cap, void* out_f16, kivi_stream_t stream) {
    const bool hs = scale_f16_of(bits);
    bits = width_of(bits);
    kivi_status st = shape_check(D, group_size, bits);
    if (st != KIVI_OK) return st;
    if ((axis != KIVI_AXIS_KEYS && axis != KIVI_AXIS_VALUES) || BH <= 0 || S < 0 || s_cap <= 0 ||
        s_cap % group_size != 0 || S > s_cap)
        return KIVI_ERR_INVALID_ARG;
    if (S == 0) return KIVI_OK;
    if (!codes_u8 || !scale || !zero_f16 || !out_f16) return KIVI_ERR_INVALID_ARG;
    if (!aligned16(codes_u8) || !aligned16(scale) || !aligned16(zero_f16) || !aligned16(out_f16))
        return KIVI_ERR_ALIGNMENT;
    DequantArgs a;
    a.codes = static_cast<const uint8_t*>(codes_u8);
    a.scale = scale;
    a.zero = static_cast<const __half*>(zero_f16);
    a.BH = BH;
    a.S = S;
    a.s_cap = s_cap;
    a.out = static_cast<__half*>(out_f16);
    a.G = group_size;
    a.D = D;
    a.scale_f16 = hs;
    return from_cuda(launch_dequant((int)axis, a, bits, reinterpret_cast<cudaStream_t>(stream)));
}

kivi_status kivi_dequant_kv(const void* kcodes_u8, const float* kscale, const void* kzero_f16,
                            const void* vcodes_u8, const float* vscale, const void* vzero_f16, int BH, int S,
                            int D, int group_size, int bits, int s_cap, void* kout_f16, void* vout_f16,
                            kivi_stream_t stream) {
    const bool hs = scale_f16_of(bits);
    bits = width_of(bits);
    kivi_status st = shape_check(D, group_size, bits);
    if (st != KIVI_OK) return st;
    if (BH <= 0 || S < 0 || s_cap <= 0 || s_cap % group_size != 0 || S > s_cap) return KIVI_ERR_INVALID_ARG;
    if (S == 0) return KIVI_OK;
    if (!kcodes_u8 || !kscale || !kzero_f16 || !vcodes_u8 || !vscale || !vzero_f16 || !kout_f16 || !vout_f16)
        return KIVI_ERR_INVALID_ARG;
    if (!aligned16(kcodes_u8) || !aligned16(kscale) || !aligned16(kzero_f16) || !aligned16(vcodes_u8) ||
        !aligned16(vscale) || !aligned16(vzero_f16) || !aligned16(kout_f16) || !aligned16(vout_f16))
        return KIVI_ERR_ALIGNMENT;
    DequantArgs k, v;
    k.codes = static_cast<const uint8_t*>(kcodes_u8);
    k.scale = kscale;
    k.zero = static_cast<const __half*>(kzero_f16);
    k.out = static_cast<__half*>(kout_f16);
    v.codes = static_cast<const uint8_t*>(vcodes_u8);
    v.scale = vscale;
    v.zero = static_cast<const __half*>(vzero_f16);
    v.out = static_cast<__half*>(vout_f16);
    k.BH = v.BH = BH;
    k.S = v.S = S;
    k.s_cap = v.s_cap = s_cap;
    k.G = v.G = group_size;
    k.D = v.D = D;
    k.scale_f16 = v.scale_f16 = hs;
    return from_cuda(launch_dequant_kv(k, v, bits, reinterpret_cast<cudaStream_t>(stream)));
}

kivi_status kivi_residual_append(const void* src_f16, int src_bh_stride, int n_new, void* res_f16,
                                 int BH, int res_cap, int D, int n_res, kivi_stream_t stream) {
    if (!head_dim_ok(D)) return KIVI_ERR_UNSUPPORTED;
    if (BH <= 0 || n_new < 0 || n_res < 0 || res_cap <= 0 || src_bh_stride < n_new ||
        (long long)n_res + n_new > res_cap)
        return KIVI_ERR_INVALID_ARG;
    if (n_new == 0) return KIVI_OK;
    if (!src_f16 || !res_f16) return KIVI_ERR_INVALID_ARG;
    if (!aligned16(src_f16) || !aligned16(res_f16)) return KIVI_ERR_ALIGNMENT;
    return from_cuda(launch_residual_append(static_cast<const __half*>(src_f16), nullptr, src_bh_stride, n_new,
                                            static_cast<__half*>(res_f16), nullptr, BH, res_cap, n_res, D,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

kivi_status kivi_residual_compact(void* res_f16, int BH, int res_cap, int D, int n_res, int n_drop,
                                  kivi_stream_t stream) {
    if (!head_dim_ok(D)) return KIVI_ERR_UNSUPPORTED;
    if (BH <= 0 || res_cap <= 0 || n_res < 0 || n_res > res_cap || n_drop < 0 || n_drop > n_res)
        return KIVI_ERR_INVALID_ARG;
    if (n_drop == 0 || n_drop == n_res) return KIVI_OK;
    if (!res_f16) return KIVI_ERR_INVALID_ARG;
    if (!aligned16(res_f16)) return KIVI_ERR_ALIGNMENT;
    return from_cuda(launch_residual_compact(static_cast<__half*>(res_f16), nullptr, BH, res_cap, n_res, n_drop, D,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

kivi_status kivi_residual_append_kv(const void* k_src_f16, const void* v_src_f16, int src_bh_stride, int n_new,
                                    void* k_res_f16, void* v_res_f16, int BH, int res_cap, int D, int n_res,
                                    kivi_stream_t stream) {
    if (!head_dim_ok(D)) return KIVI_ERR_UNSUPPORTED;
    if (BH <= 0 || n_new < 0 || n_res < 0 || res_cap <= 0 || src_bh_stride < n_new ||
        (long long)n_res + n_new > res_cap)
        return KIVI_ERR_INVALID_ARG;
    if (n_new == 0) return KIVI_OK;
    if (!k_src_f16 || !v_src_f16 || !k_res_f16 || !v_res_f16) return KIVI_ERR_INVALID_ARG;
    if (!aligned16(k_src_f16) || !aligned16(v_src_f16) || !aligned16(k_res_f16) || !aligned16(v_res_f16))
        return KIVI_ERR_ALIGNMENT;
    return from_cuda(launch_residual_append(static_cast<const __half*>(k_src_f16),
                                            static_cast<const __half*>(v_src_f16), src_bh_stride, n_new,
                                            static_cast<__half*>(k_res_f16), static_cast<__half*>(v_res_f16), BH,
                                            res_cap, n_res, D, reinterpret_cast<cudaStream_t>(stream)));
}

kivi_status kivi_residual_compact_kv(void* k_res_f16, void* v_res_f16, int BH, int res_cap, int D, int n_res,
                                     int n_drop, kivi_stream_t stream) {
    if (!head_dim_ok(D)) return KIVI_ERR_UNSUPPORTED;
    if (BH <= 0 || res_cap <= 0 || n_res < 0 || n_res > res_cap || n_drop < 0 || n_drop > n_res)
        return KIVI_ERR_INVALID_ARG;
    if (n_drop == 0 || n_drop == n_res) return KIVI_OK;
    if (!k_res_f16 || !v_res_f16) return KIVI_ERR_INVALID_ARG;
    if (!aligned16(k_res_f16) || !aligned16(v_res_f16)) return KIVI_ERR_ALIGNMENT;
    return from_cuda(launch_residual_compact(static_cast<__half*>(k_res_f16), static_cast<__half*>(v_res_f16), BH,
                                             res_cap, n_res, n_drop, D, reinterpret_cast<cudaStream_t>(stream)));
}

size_t kivi_decode_workspace_size(int B, int Hq, int Hkv, int S_q, int n_res, int D) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || S_q < 0 || n_res < 0 || !head_dim_ok(D) || S_q + n_res == 0)
        return 0;
    // the plan depends on the bit width and, through the choice of kernel, on
    // the group size; the size covers every plan
    size_t w = 0;
    for (int bits : {2, 4})
        for (bool pair_ok : {false, true}) {
            const size_t wb = workspace_bytes(B, Hq, D, make_plan(B, Hkv, Hq, S_q, n_res, bits, pair_ok && D == kD, D));
            if (wb > w) w = wb;
        }
    return w;
}

kivi_status kivi_decode_plan_info(int B, int Hq, int Hkv, int S_q, int n_res, int D, int group_size, int bits,
                                  int* info) {
    bits = decode_bits(bits);
    const bool hs = scale_f16_of(bits);
    bits = width_of(bits);
    kivi_status st = shape_check(D, group_size, bits);
    if (st != KIVI_OK) return st;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || S_q < 0 || n_res < 0 || S_q + n_res == 0)
        return KIVI_ERR_INVALID_ARG;
    if (Hq / Hkv > 64) return KIVI_ERR_UNSUPPORTED;
    if (!info) return KIVI_ERR_INVALID_ARG;
    // the plan kivi_decode_attend takes for these arguments
    const DecodePlan p = make_plan(B, Hkv, Hq, S_q, n_res, bits, group_size == kG && D == kD && !hs, D);
    info[0] = p.pair_kernel;
    info[1] = p.n_split;
    info[2] = p.tiles_per_warp;
    info[3] = p.pair_kernel ? 2 * kPairsPerCta : p.warps_per_cta;
    info[4] = p.q_sub;
    info[5] = p.n_tiles;
    info[6] = p.tiles_per_split;
    return KIVI_OK;
}

kivi_status kivi_decode_attend(const void* q_f16, const void* kcodes_u8, const float* kscale,
                               const void* kzero_f16, const void* vcodes_u8, const float* vscale,
                               const void* vzero_f16, int S_q, int s_cap, const void* k_res_f16,
                               const void* v_res_f16, int n_res, int res_cap, int B, int Hq, int Hkv,
                               int D, int group_size, int bits, float sm_scale, float* out_f32,
                               void* workspace, size_t workspace_bytes_, kivi_stream_t stream) {
    const bool ready = store_ready_of(bits);
    bits = decode_bits(bits);
    const bool hs = scale_f16_of(bits);
    bits = width_of(bits);
    kivi_status st = shape_check(D, group_size, bits);
    if (st != KIVI_OK) return st;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || S_q < 0 || n_res < 0 ||
        S_q + n_res == 0 || S_q > s_cap || n_res > res_cap || s_cap < 0 || res_cap < 0 ||
        (S_q > 0 && s_cap % group_size != 0) || !std::isfinite(sm_scale))
        return KIVI_ERR_INVALID_ARG;
    const int gq = Hq / Hkv;
    if (gq > 64) return KIVI_ERR_UNSUPPORTED;  // up to 16 sub-groups of 4 query heads
    if (!q_f16 || !out_f32) return KIVI_ERR_INVALID_ARG;
    if (S_q > 0 && (!kcodes_u8 || !kscale || !kzero_f16 || !vcodes_u8 || !vscale || !vzero_f16))
        return KIVI_ERR_INVALID_ARG;
    if (n_res > 0 && (!k_res_f16 || !v_res_f16)) return KIVI_ERR_INVALID_ARG;
    if (!aligned16(q_f16) || !aligned16(out_f32) || !aligned16(kcodes_u8) || !aligned16(kscale) ||
        !aligned16(kzero_f16) || !aligned16(vcodes_u8) || !aligned16(vscale) ||
        !aligned16(vzero_f16) || !aligned16(k_res_f16) || !aligned16(v_res_f16) ||
        !aligned16(workspace))
        return KIVI_ERR_ALIGNMENT;
    const DecodePlan p = make_plan(B, Hkv, Hq, S_q, n_res, bits, group_size == kG && D == kD && !hs, D);
    const size_t need = workspace_bytes(B, Hq, D, p);
    if (need > 0 && (!workspace || workspace_bytes_ < need)) return KIVI_ERR_WORKSPACE;

    DecodeArgs a;
    a.q = static_cast<const __half*>(q_f16);
    a.kcodes = static_cast<const uint8_t*>(kcodes_u8);
    a.kscale = kscale;
    a.kzero = static_cast<const __half*>(kzero_f16);
    a.vcodes = static_cast<const uint8_t*>(vcodes_u8);
    a.vscale = vscale;
    a.vzero = static_cast<const __half*>(vzero_f16);
    a.S_q = S_q;
    a.s_cap = s_cap;
    a.g_shift = group_size == 128 ? 2 : (group_size == 64 ? 1 : 0);
    a.D = D;
    a.scale_f16 = hs ? 1 : 0;
    a.k_res = static_cast<const __half*>(k_res_f16);
    a.v_res = static_cast<const __half*>(v_res_f16);
    a.n_res = n_res;
    a.res_cap = res_cap;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.score_scale = sm_scale * 1.4426950408889634f;
    a.n_split = p.n_split;
    a.tiles_per_split = p.tiles_per_split;
    a.tiles_per_warp = p.tiles_per_warp;
    a.warps_per_cta = p.warps_per_cta;
    a.pair_kernel = p.pair_kernel;
    a.n_store_tiles = p.n_store_tiles;
    a.n_tiles = p.n_tiles;
    char* ws = static_cast<char*>(workspace);
    a.counters = need > 0 ? reinterpret_cast<unsigned int*>(ws) : nullptr;
    a.part_o = need > 0 ? reinterpret_cast<float*>(ws + KIVI_DECODE_COUNTER_BYTES) : nullptr;
    a.part_ml = need > 0 ? reinterpret_cast<float*>(ws + KIVI_DECODE_COUNTER_BYTES + part_o_bytes(B, Hq, D, p))
                         : nullptr;
    a.out = out_f32;
    const cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);
    a.q_sub = p.q_sub;
    a.store_ready = ready ? 1 : 0;
    return from_cuda(p.pair_kernel ? launch_decode_pair(a, bits, gq, strm) : launch_decode_mma(a, bits, gq, strm));
}

kivi_status kivi_decode_workspace_init(void* workspace, size_t workspace_bytes_, kivi_stream_t stream) {
    if (workspace_bytes_ == 0) return KIVI_OK;
    if (!workspace) return KIVI_ERR_INVALID_ARG;
    const size_t n = workspace_bytes_ < (size_t)KIVI_DECODE_COUNTER_BYTES ? workspace_bytes_
                                                                         : (size_t)KIVI_DECODE_COUNTER_BYTES;
    return from_cuda(cudaMemsetAsync(workspace, 0, n, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
