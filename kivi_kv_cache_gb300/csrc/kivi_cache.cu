// kivi_cache.cu -- one attention layer's KIVI cache as a host-side state
// machine over the library's entry points: kivi_cache_prefill,
// kivi_cache_append and kivi_cache_decode (declared in include/kivi.h).
//
// Method: VeloxQuant-MLX blog, "A 5.65x Metal Kernel That Made My LLM Exactly
// 0% Faster", "What we're actually optimizing": the newest residual_length
// tokens stay in fp16, and once the window has grown a group of G past that,
// its oldest whole groups are quantized into the packed store; the section
// "Four benchmarks that lied" (Lie #2) counts those flushes per decode run.
// The rule: whenever the window holds n_res >= R + G tokens, its oldest
// floor((n_res - R) / G) * G tokens are flushed at store offset S_q, so
// R <= n_res < R + G afterwards. The window is rows res_off .. res_off +
// n_res - 1 of its buffer: a flush advances res_off, and the remaining
// tokens move back to row 0 only when an append would not fit behind them.
//
// Every step runs in the library's kernels (residual append, flush, residual
// compact, decode); this file only sequences them and keeps the counters.
// All argument checks run before the first launch of a call: a call that
// fails a check launches nothing and leaves the counters as they were.
#include "../../include/kivi.h"
#include "kivi_launch.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Geometry, buffers and counters of a cache, before any launch.
kivi_status cache_check(const kivi_cache* c) {
    if (!c) return KIVI_ERR_INVALID_ARG;
    if (c->group_size <= 0 || c->D <= 0) return KIVI_ERR_INVALID_ARG;
    const kivi_status sh = static_cast<kivi_status>(kivi::shape_status(c->D, c->group_size, c->bits));
    if (sh != KIVI_OK) return sh;
    if (c->BH <= 0 || c->residual_length < 0 || c->s_cap <= 0 || c->s_cap % c->group_size != 0 ||
        (long long)c->res_cap < (long long)c->residual_length + c->group_size || c->S_q < 0 || c->S_q > c->s_cap ||
        c->n_res < 0 || c->res_off < 0 || (long long)c->res_off + c->n_res > c->res_cap)
        return KIVI_ERR_INVALID_ARG;
    const void* bufs[8] = {c->kcodes, c->kscale, c->kzero, c->vcodes, c->vscale, c->vzero, c->k_res, c->v_res};
    for (const void* p : bufs) {
        if (!p) return KIVI_ERR_INVALID_ARG;
        if (!aligned16(p)) return KIVI_ERR_ALIGNMENT;
    }
    return KIVI_OK;
}

// Tokens a window of n_res tokens flushes: floor((n_res - R) / G) * G once
// n_res >= R + G, else 0.
int window_flush(int n_res, int R, int G) { return n_res >= R + G ? (n_res - R) / G * G : 0; }

// Row r of the window buffers (16-byte aligned: rows are 2 D bytes, D >= 64).
const void* window_row(const void* base, const kivi_cache* c, int r) {
    return static_cast<const __half*>(base) + (long long)r * c->D;
}

// Flush the oldest n tokens of the windows into the stores at S_q (exactly n:
// the windows are passed from row res_off as n tokens with residual_length
// 0); the window then starts n rows later.
kivi_status flush_window(kivi_cache* c, int n, kivi_stream_t stream) {
    int done = 0;
    kivi_status st = kivi_flush_kv(window_row(c->k_res, c, c->res_off), window_row(c->v_res, c, c->res_off), c->BH,
                                   n, c->res_cap, c->D, c->group_size, c->bits, 0, c->kcodes, c->kscale, c->kzero,
                                   c->vcodes, c->vscale, c->vzero, c->S_q, c->s_cap, &done, stream);
    if (st != KIVI_OK) return st;
    c->S_q += done;
    c->store_written = 1;
    c->n_res -= done;
    c->res_off = c->n_res == 0 ? 0 : c->res_off + done;
    return KIVI_OK;
}

// Move the window's n_res tokens from row res_off to row 0 (an overlap-safe
// copy) so that m more tokens fit behind them; nothing to do if they fit.
kivi_status make_room(kivi_cache* c, int m, kivi_stream_t stream) {
    if ((long long)c->res_off + c->n_res + m <= c->res_cap || c->res_off == 0) return KIVI_OK;
    const kivi_status st = kivi_residual_compact_kv(c->k_res, c->v_res, c->BH, c->res_cap, c->D,
                                                    c->res_off + c->n_res, c->res_off, stream);
    if (st != KIVI_OK) return st;
    c->res_off = 0;
    if (c->n_res > 0) c->store_written = 0;
    return KIVI_OK;
}

}  // namespace

extern "C" {

kivi_status kivi_cache_prefill(kivi_cache* c, const void* k_f16, const void* v_f16, int x_bh_stride, int S,
                               int* n_flushed, kivi_stream_t stream) {
    kivi_status st = cache_check(c);
    if (st != KIVI_OK) return st;
    if (c->n_res != 0 || S < 0 || x_bh_stride < S) return KIVI_ERR_INVALID_ARG;
    const int G = c->group_size;
    const int n = kivi_flush_count(S, c->residual_length, G);
    const int tail = S - n;
    if ((long long)c->S_q + n > c->s_cap || tail > c->res_cap || (n > 0 && c->S_q % G != 0))
        return KIVI_ERR_INVALID_ARG;
    if (S > 0 && (!k_f16 || !v_f16)) return KIVI_ERR_INVALID_ARG;
    if (S > 0 && (!aligned16(k_f16) || !aligned16(v_f16))) return KIVI_ERR_ALIGNMENT;
    if (n_flushed) *n_flushed = 0;
    if (n > 0) {
        int done = 0;
        st = kivi_flush_kv(k_f16, v_f16, c->BH, S, x_bh_stride, c->D, G, c->bits, c->residual_length, c->kcodes,
                           c->kscale, c->kzero, c->vcodes, c->vscale, c->vzero, c->S_q, c->s_cap, &done, stream);
        if (st != KIVI_OK) return st;
        c->S_q += done;
        c->store_written = 1;
        if (n_flushed) *n_flushed = done;
    }
    if (tail > 0) {
        const __half* k = static_cast<const __half*>(k_f16) + (long long)n * c->D;
        const __half* v = static_cast<const __half*>(v_f16) + (long long)n * c->D;
        st = kivi_residual_append_kv(k, v, x_bh_stride, tail, c->k_res, c->v_res, c->BH, c->res_cap, c->D, 0,
                                     stream);
        if (st != KIVI_OK) return st;
        c->n_res = tail;
        c->store_written = 0;
    }
    c->res_off = 0;
    return KIVI_OK;
}

kivi_status kivi_cache_append(kivi_cache* c, const void* k_f16, const void* v_f16, int src_bh_stride, int n_new,
                              int* n_flushed, kivi_stream_t stream) {
    kivi_status st = cache_check(c);
    if (st != KIVI_OK) return st;
    if (n_new < 0 || src_bh_stride < n_new) return KIVI_ERR_INVALID_ARG;
    if (n_flushed) *n_flushed = 0;
    if (n_new == 0) return KIVI_OK;
    if (!k_f16 || !v_f16) return KIVI_ERR_INVALID_ARG;
    if (!aligned16(k_f16) || !aligned16(v_f16)) return KIVI_ERR_ALIGNMENT;
    const int R = c->residual_length, G = c->group_size;
    // Dry run on the counters: the new tokens enter in pieces that fit the
    // window (the whole batch when res_cap >= R + G + n_new), each piece
    // followed by the flush it triggers. Every store offset must stay a
    // multiple of G and within the store.
    {
        long long S_q = c->S_q;
        int n_res = c->n_res, left = n_new;
        while (left > 0) {
            const int m = left < c->res_cap - n_res ? left : c->res_cap - n_res;
            if (m <= 0) return KIVI_ERR_INVALID_ARG;  // unreachable: a flush leaves n_res < R + G <= res_cap
            n_res += m;
            left -= m;
            const int f = window_flush(n_res, R, G);
            if (f > 0) {
                if (S_q % G != 0 || S_q + f > c->s_cap) return KIVI_ERR_INVALID_ARG;
                S_q += f;
                n_res -= f;
            }
        }
    }
    int flushed = 0, off = 0;
    while (off < n_new) {
        const int room = c->res_cap - c->n_res;
        const int m = n_new - off < room ? n_new - off : room;
        st = make_room(c, m, stream);
        if (st != KIVI_OK) return st;
        const __half* k = static_cast<const __half*>(k_f16) + (long long)off * c->D;
        const __half* v = static_cast<const __half*>(v_f16) + (long long)off * c->D;
        st = kivi_residual_append_kv(k, v, src_bh_stride, m, c->k_res, c->v_res, c->BH, c->res_cap, c->D,
                                     c->res_off + c->n_res, stream);
        if (st != KIVI_OK) return st;
        c->n_res += m;
        c->store_written = 0;
        off += m;
        const int f = window_flush(c->n_res, R, G);
        if (f > 0) {
            st = flush_window(c, f, stream);
            if (st != KIVI_OK) return st;
            flushed += f;
            if (n_flushed) *n_flushed = flushed;
        }
    }
    return KIVI_OK;
}

kivi_status kivi_cache_decode(const kivi_cache* c, const void* q_f16, int B, int Hq, int Hkv, float sm_scale,
                              float* out_f32, void* workspace, size_t workspace_bytes, kivi_stream_t stream) {
    kivi_status st = cache_check(c);
    if (st != KIVI_OK) return st;
    if (B <= 0 || Hkv <= 0 || (long long)B * Hkv != c->BH) return KIVI_ERR_INVALID_ARG;
    const int bits = c->bits | (c->store_written ? 0 : KIVI_DECODE_STORE_READY);
    return kivi_decode_attend(q_f16, c->kcodes, c->kscale, c->kzero, c->vcodes, c->vscale, c->vzero, c->S_q,
                              c->s_cap, window_row(c->k_res, c, c->res_off), window_row(c->v_res, c, c->res_off),
                              c->n_res, c->res_cap, B, Hq, Hkv, c->D, c->group_size, bits, sm_scale, out_f32,
                              workspace, workspace_bytes, stream);
}

}  // extern "C"
