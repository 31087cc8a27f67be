// api.cu -- the C ABI of libmercury_attn.so: argument validation, status
// codes and messages, the shift planner, and dispatch to the kernels.
// Declarations and the full contract are in include/mercury_attn.h.
#include <cuda_runtime.h>

#include <limits.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "internal.h"
#include "work.h"

using namespace mercury;

namespace {

thread_local char g_msg[512];

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return code;
}

int ok()
{
    g_msg[0] = '\0';
    return MERCURY_OK;
}

bool aligned(const void *p, uintptr_t a)
{
    return ((uintptr_t)p % a) == 0;
}

unsigned long long wait_budget_ns()
{
    const char *e = getenv("MERCURY_WAIT_NS");
    if (e && *e) {
        char *end = nullptr;
        unsigned long long v = strtoull(e, &end, 10);
        if (end && *end == '\0' && v > 0)
            return v;
    }
    return 2000000000ull;  // 2 s
}

int fault_mode()
{
    const char *e = getenv("MERCURY_FAULT");
    if (e && strcmp(e, "drop_p_arrive") == 0)
        return 1;
    return 0;
}

bool sync_check()
{
    const char *e = getenv("MERCURY_SYNC_CHECK");
    return e && e[0] == '1';
}

// Overflow-checked product of non-negative factors; false if > 2^62.
bool mul_ok(long long &acc, long long f)
{
    if (f < 0)
        return false;
    if (f != 0 && acc > (1LL << 62) / f)
        return false;
    acc *= f;
    return true;
}

int check_shift(int R, int shift)
{
    if (R < 1 || R > kMaxR)
        return fail(MERCURY_EINVAL, "R must be in [1, %d] (got %d)", kMaxR, R);
    if (shift < 0)
        return fail(MERCURY_EINVAL, "shift must be >= 0 (got %d)", shift);
    if (shift >= 2 && R % shift != 0)
        return fail(MERCURY_EINVAL, "nested shift: inner size %d must divide R = %d", shift, R);
    return MERCURY_OK;
}

int check_attn_args(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq, int Skv,
                    int d, int R, int shift, int causal, const float *out, const float *lse, int partial)
{
    if (!q || !k || !v || !out || !lse)
        return fail(MERCURY_EINVAL, "null pointer argument");
    if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Skv < 1)
        return fail(MERCURY_EINVAL, "B, Hq, Hkv, Sq, Skv must be >= 1");
    if (Hq % Hkv != 0)
        return fail(MERCURY_EINVAL, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
    if (d != 64 && d != 128)
        return fail(MERCURY_EINVAL, "head dim must be 64 or 128 (got %d)", d);
    int rc = check_shift(R, shift);
    if (rc)
        return rc;
    if (Sq % R != 0 || Skv % R != 0)
        return fail(MERCURY_EINVAL, "R (%d) must divide Sq (%d) and Skv (%d)", R, Sq, Skv);
    if (causal && Sq > Skv)
        return fail(MERCURY_EINVAL, "causal attention needs Sq <= Skv (Sq %d, Skv %d)", Sq, Skv);
    long long nq = 1, nkv = 1;
    if (!mul_ok(nq, B) || !mul_ok(nq, Hq) || !mul_ok(nq, Sq) || !mul_ok(nq, d) ||
        (partial && !mul_ok(nq, R)) || !mul_ok(nkv, B) || !mul_ok(nkv, Hkv) || !mul_ok(nkv, Skv) ||
        !mul_ok(nkv, d))
        return fail(MERCURY_EINVAL, "tensor sizes overflow");
    if ((long long)B * Hq > INT_MAX || (long long)B * Hkv > INT_MAX)
        return fail(MERCURY_EINVAL, "B*H exceeds 2^31");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
        return fail(MERCURY_EALIGN, "q, k, v and the O output must be 16-byte aligned");
    if (!aligned(lse, 4))
        return fail(MERCURY_EALIGN, "the LSE output must be 4-byte aligned");
    return MERCURY_OK;
}

int finish(int rc, cudaStream_t stream)
{
    if (rc != MERCURY_OK)
        return rc;
    if (sync_check()) {
        unsigned int w = 0, site = 0;
        rc = read_and_clear_device_error(stream, &w, &site, g_msg, sizeof g_msg);
        if (rc != MERCURY_OK)
            return rc;
        if (w & 1u)
            return fail(MERCURY_ETIMEOUT, "a bounded device wait ran out (site 0x%x)", site);
    }
    return ok();
}

int attn_common(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq, int Skv,
                int d, int R, int shift, int causal, float *out, float *lse, void *stream, int partial)
{
    int rc = check_attn_args(q, k, v, B, Hq, Hkv, Sq, Skv, d, R, shift, causal, out, lse, partial);
    if (rc)
        return rc;
    int order[kMaxR * kMaxR];
    if (plan_shift(R, shift, order))
        return fail(MERCURY_EINVAL, "invalid (R, shift)");
    AttnCall c;
    c.q = q;
    c.k = k;
    c.v = v;
    c.B = B;
    c.Hq = Hq;
    c.Hkv = Hkv;
    c.Sq = Sq;
    c.Skv = Skv;
    c.d = d;
    c.R = R;
    c.causal = causal ? 1 : 0;
    c.partial = partial;
    c.order = order;
    c.out = out;
    c.lse = lse;
    c.wait_ns = wait_budget_ns();
    c.fault = fault_mode();
    cudaStream_t s = (cudaStream_t)stream;
    rc = launch_attention(c, s, g_msg, sizeof g_msg);
    return finish(rc, s);
}

}  // namespace

extern "C" {

int mercury_plan_shift(int R, int shift, int *order)
{
    if (!order)
        return fail(MERCURY_EINVAL, "order is NULL");
    int rc = check_shift(R, shift);
    if (rc)
        return rc;
    if (plan_shift(R, shift, order))
        return fail(MERCURY_EINVAL, "invalid (R, shift)");
    return ok();
}

int mercury_attn_sharded(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq, int Skv,
                         int d, int R, int shift, int causal, float *out, float *lse, void *stream)
{
    return attn_common(q, k, v, B, Hq, Hkv, Sq, Skv, d, R, shift, causal, out, lse, stream, 0);
}

int mercury_attn_partial(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq, int Skv,
                         int d, int R, int shift, int causal, float *o_part, float *lse_part, void *stream)
{
    return attn_common(q, k, v, B, Hq, Hkv, Sq, Skv, d, R, shift, causal, o_part, lse_part, stream, 1);
}

int mercury_lse_merge(const float *o_part, const float *lse_part, int n_parts, long long rows, int d,
                      float *out, float *lse, void *stream)
{
    if (!o_part || !lse_part || !out || !lse)
        return fail(MERCURY_EINVAL, "null pointer argument");
    if (n_parts < 1 || n_parts > 4096)
        return fail(MERCURY_EINVAL, "n_parts must be in [1, 4096] (got %d)", n_parts);
    if (rows < 0)
        return fail(MERCURY_EINVAL, "rows must be >= 0");
    if (d < 4 || d > 512 || d % 4 != 0)
        return fail(MERCURY_EINVAL, "d must be a multiple of 4 in [4, 512] (got %d)", d);
    long long n = 1;
    if (!mul_ok(n, n_parts) || !mul_ok(n, rows) || !mul_ok(n, d))
        return fail(MERCURY_EINVAL, "tensor sizes overflow");
    if (!aligned(o_part, 16) || !aligned(out, 16))
        return fail(MERCURY_EALIGN, "o_part and out must be 16-byte aligned");
    if (!aligned(lse_part, 4) || !aligned(lse, 4))
        return fail(MERCURY_EALIGN, "lse_part and lse must be 4-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    int rc = launch_lse_merge(o_part, lse_part, n_parts, rows, d, out, lse, s, g_msg, sizeof g_msg);
    return finish(rc, s);
}

int mercury_sync_status(void *stream)
{
    unsigned int w = 0, site = 0;
    int rc = read_and_clear_device_error((cudaStream_t)stream, &w, &site, g_msg, sizeof g_msg);
    if (rc != MERCURY_OK)
        return rc;
    if (w & 1u)
        return fail(MERCURY_ETIMEOUT, "a bounded device wait ran out (site 0x%x)", site);
    return ok();
}

const char *mercury_last_error(void)
{
    return g_msg;
}

int mercury_work_decomposition(int B, int Hq, int Hkv, int Sq, int Skv, int d, int R, int causal, int partial,
                               long long *info)
{
    if (!info)
        return fail(MERCURY_EINVAL, "info is NULL");
    if (d != 64 && d != 128)
        return fail(MERCURY_EINVAL, "head dim must be 64 or 128 (got %d)", d);
    if (causal && Sq > Skv)
        return fail(MERCURY_EINVAL, "causal attention needs Sq <= Skv");
    Geom g;
    if (make_geom(g, B, Hq, Hkv, Sq, Skv, d, R, causal, partial))
        return fail(MERCURY_EINVAL, "unsupported shape");
    info[0] = g.Mq;
    info[1] = g.Gp;
    info[2] = g.head_mode;
    info[3] = g.T_h;
    info[4] = g.T_r;
    info[5] = (long long)g.NHP * g.NRT;
    info[6] = g.n_items;
    info[7] = 0;
    return ok();
}

int mercury_work_item_rows(int B, int Hq, int Hkv, int Sq, int Skv, int d, int R, int shift, int causal,
                           int partial, long long item, long long *rows, int *n_rows, int *step)
{
    if (!rows || !n_rows || !step)
        return fail(MERCURY_EINVAL, "null pointer argument");
    if (d != 64 && d != 128)
        return fail(MERCURY_EINVAL, "head dim must be 64 or 128 (got %d)", d);
    if (causal && Sq > Skv)
        return fail(MERCURY_EINVAL, "causal attention needs Sq <= Skv");
    int rc = check_shift(R, shift);
    if (rc)
        return rc;
    Geom g;
    if (make_geom(g, B, Hq, Hkv, Sq, Skv, d, R, causal, partial))
        return fail(MERCURY_EINVAL, "unsupported shape");
    if (item < 0 || item >= g.n_items)
        return fail(MERCURY_EINVAL, "item out of range");
    int order[kMaxR * kMaxR];
    plan_shift(R, shift, order);
    Item it = decode_item(g, item);
    int n = 0;
    for (int t = 0; t < 2; ++t) {
        if (!it.t[t].valid)
            continue;
        for (int r = 0; r < kTileRows; ++r) {
            if (r % g.Mq >= it.t[t].nq)
                continue;
            const long long head = it.t[t].h0 + r / g.Mq;
            const long long qi = it.t[t].q0 + r % g.Mq;
            rows[n++] = ((long long)it.b * Hq + head) * Sq + qi;
        }
    }
    *n_rows = n;
    *step = -1;
    if (partial) {
        for (int j = 0; j < R; ++j)
            if (order[it.rank * R + j] == it.shard)
                *step = j;
    }
    return ok();
}

}  // extern "C"
