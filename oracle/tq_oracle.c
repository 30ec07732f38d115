/*
 * tq_oracle.c -- plain, slow CPU oracle for the TurboQuant KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY (see tq_oracle.h).  Compiled with
 * -ffp-contract=off so every float/double operation is one IEEE rounding.
 * Every function cites the page passage it restates.
 */
#include "tq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

/* ======================================================================
 * Layout.  [vLLM-API] "__init__": key data bytes = ceil(D * mse_bits / 8)
 * for MSE keys, D for fp8 keys; value data bytes = ceil(D * vbits / 8).
 * [vLLM-API] "_continuation_prefill": metadata fields k_norm (MSE only),
 * v_scale, v_zero, each fp16.  [vLLM-PR] "turboquant_attn.py"
 * get_kv_cache_shape: slot rounded up to an even byte count.
 * Presets: [vLLM-PR] "turboquant_attn.py" supported_kv_cache_dtypes and
 * the "k8v4 = FP8 keys + 4-bit values" discussion in the review notes.
 * ==================================================================== */
int orc_get_layout(int preset, int D, orc_layout* L)
{
    if (!L || D <= 0) return -1;
    if (preset & ~(0xFF | ORC_LAYOUT_SOA)) return -1;
    memset(L, 0, sizeof(*L));
    switch (preset & 0xFF) {
    case ORC_K8V4:    L->key_fp8 = 1; L->key_bits = 8; L->value_bits = 4; L->norm_correction = 0; break;
    case ORC_4BIT_NC: L->key_fp8 = 0; L->key_bits = 4; L->value_bits = 4; L->norm_correction = 1; break;
    case ORC_K3V4_NC: L->key_fp8 = 0; L->key_bits = 3; L->value_bits = 4; L->norm_correction = 1; break;
    case ORC_3BIT_NC: L->key_fp8 = 0; L->key_bits = 3; L->value_bits = 3; L->norm_correction = 1; break;
    case ORC_2BIT_NC: L->key_fp8 = 0; L->key_bits = 2; L->value_bits = 2; L->norm_correction = 1; break;
    default: return -1;
    }
    int pos = 0;
    if (L->key_fp8) {
        L->key_data_bytes = D;
        pos = D;
        L->off_k_norm = -1;
    } else {
        L->key_data_bytes = (D * L->key_bits + 7) / 8;
        pos = L->key_data_bytes;
        L->off_k_norm = pos;
        pos += 2;
    }
    L->off_v_data = pos;
    L->value_data_bytes = (D * L->value_bits + 7) / 8;
    pos += L->value_data_bytes;
    L->off_v_scale = pos; pos += 2;
    L->off_v_zero = pos;  pos += 2;
    L->slot_size = pos;
    L->slot_size_aligned = ((pos + 1) / 2) * 2;
    return 0;
}

/* ======================================================================
 * Scalar formats, each from its published definition.
 * ==================================================================== */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double orc_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0)       v = ldexp((double)f, -24);
    else if (e == 31) v = f ? NAN : INFINITY;
    else              v = ldexp(1.0 + f / 1024.0, e - 15);
    return sign ? -v : v;
}

/* Round-to-nearest-even of a double to binary16; overflow -> inf. */
uint16_t orc_double_to_f16(double x)
{
    if (isnan(x)) return 0x7E00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a >= 65520.0) return sign | 0x7C00;          /* rounds past 65504 */
    if (a < ldexp(1.0, -14)) {                        /* subnormal range   */
        double q = nearbyint(a * ldexp(1.0, 24));     /* units of 2^-24    */
        return sign | (uint16_t)q;                    /* q==1024 -> min normal */
    }
    int E;
    frexp(a, &E);                                     /* a = f*2^E, f in [.5,1) */
    int e = E - 1;                                    /* a in [2^e, 2^(e+1))    */
    double q = nearbyint((ldexp(a, -e) - 1.0) * 1024.0);
    if (q == 1024.0) { q = 0.0; e += 1; }
    if (e + 15 >= 31) return sign | 0x7C00;
    return sign | (uint16_t)(((e + 15) << 10) | (int)q);
}

/* bfloat16 is the top half of a binary32. */
float orc_bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* OCP 8-bit E4M3 ("fn"): bias 7, no infinities, S.1111.111 is NaN, max
 * finite 448.  Round to nearest even; finite values beyond the range
 * saturate to +-448 (the saturating conversion the fp8 key store uses). */
uint8_t orc_e4m3_encode(double x)
{
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {                         /* subnormals: m*2^-9 */
        double q = nearbyint(a * 512.0);
        return sign | (uint8_t)q;                     /* q==8 -> min normal */
    }
    int E;
    frexp(a, &E);
    int e = E - 1;
    double q = nearbyint((ldexp(a, -e) - 1.0) * 8.0);
    if (q == 8.0) { q = 0.0; e += 1; }
    return sign | (uint8_t)(((e + 7) << 3) | (int)q);
}

double orc_e4m3_decode(uint8_t b)
{
    int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) v = NAN;
    else if (e == 0)       v = ldexp((double)m, -9);
    else                   v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* ======================================================================
 * Lloyd-Max codebook.  [vLLM-PR] "centroids.py": solve_lloyd_max(d, bits)
 * for N(0, 1/d).  Start from the midpoints of 2^bits equal cells on
 * [-3.5 sigma, 3.5 sigma]; each iteration takes boundaries as neighbour
 * means, outer edges at 3x the init range, and replaces every centroid by
 * its cell's conditional mean, both integrals by the trapezoid rule with
 * n = 200 panels.  Stop once the largest centroid move is below tol; on
 * that exit the centroids of the previous iterate are the ones kept.
 * Cells with almost no mass (denominator <= 1e-15) keep their centroid.
 * ==================================================================== */
static double orc_pdf(double x, double sigma2)
{
    return (1.0 / sqrt(2 * M_PI * sigma2)) * exp(-x * x / (2 * sigma2));
}

/* trapezoid rule over [a, b] with n panels of f(x) = x^moment * pdf(x) */
static double orc_trapz(int moment, double a, double b, int n, double sigma2)
{
    double h = (b - a) / n;
    double fa = orc_pdf(a, sigma2), fb = orc_pdf(b, sigma2);
    if (moment) { fa = a * fa; fb = b * fb; }
    double acc = 0.5 * (fa + fb);
    for (int i = 1; i < n; ++i) {
        double x = a + i * h;
        double f = orc_pdf(x, sigma2);
        acc += moment ? x * f : f;
    }
    return acc * h;
}

int orc_lloyd_max(int d, int bits, int trapz_n, int max_iter, double tol,
                  double* centroids64, float* c32, float* m32)
{
    if (d <= 0 || bits < 1 || bits > 8 || trapz_n < 1) return -1;
    const int L = 1 << bits;
    const double sigma2 = 1.0 / d;
    const double sigma = sqrt(sigma2);
    const double lo = -3.5 * sigma, hi = 3.5 * sigma;
    double* c = (double*)malloc(sizeof(double) * L);
    double* nc = (double*)malloc(sizeof(double) * L);
    double* edge = (double*)malloc(sizeof(double) * (L + 1));
    for (int i = 0; i < L; ++i) c[i] = lo + (hi - lo) * (i + 0.5) / L;

    int it = 0;
    for (; it < max_iter; ++it) {
        edge[0] = lo * 3;
        edge[L] = hi * 3;
        for (int i = 0; i + 1 < L; ++i) edge[i + 1] = (c[i] + c[i + 1]) / 2.0;
        double move = 0.0;
        for (int i = 0; i < L; ++i) {
            double num = orc_trapz(1, edge[i], edge[i + 1], trapz_n, sigma2);
            double den = orc_trapz(0, edge[i], edge[i + 1], trapz_n, sigma2);
            nc[i] = den > 1e-15 ? num / den : c[i];
            double dm = fabs(nc[i] - c[i]);
            if (dm > move) move = dm;
        }
        if (move < tol) break;          /* keep c, the previous iterate */
        memcpy(c, nc, sizeof(double) * L);
    }
    if (centroids64) memcpy(centroids64, c, sizeof(double) * L);
    if (c32)
        for (int i = 0; i < L; ++i) c32[i] = (float)c[i];
    if (m32) {
        /* [vLLM-API] "_ensure_on_device": midpoints of the sorted fp32
         * centroids, computed in fp32 (the sum rounds once, halving is exact) */
        for (int i = 0; i + 1 < L; ++i) {
            float a = (float)c[i], b = (float)c[i + 1];
            float s = a + b;
            m32[i] = s / 2.0f;
        }
    }
    free(c); free(nc); free(edge);
    return it;
}

/* ======================================================================
 * Rotation.  [Atlas] "Background": the randomized Hadamard transform is a
 * random sign vector followed by a Walsh-Hadamard transform.
 * [vLLM-API] "_ensure_on_device": H is the orthonormal, symmetric
 * Hadamard matrix (H = H^T, H H = I).  The sign generator is not given on
 * the pages; this oracle uses SplitMix64 (Steele, Lea & Flood, OOPSLA
 * 2014), whose i-th output from state `seed` is mix(seed + (i+1)*gamma).
 * ==================================================================== */
static uint64_t orc_splitmix64_at(uint64_t seed, uint64_t i)
{
    uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

void orc_signs(int D, uint64_t seed, int8_t* s)
{
    for (int i = 0; i < D; ++i)
        s[i] = (orc_splitmix64_at(seed, (uint64_t)i) >> 63) ? -1 : 1;
}

static int orc_popcount(unsigned x)
{
    int n = 0;
    while (x) { n += x & 1u; x >>= 1; }
    return n;
}

void orc_hadamard(int D, double* H)
{
    double r = 1.0 / sqrt((double)D);
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j)
            H[(size_t)i * D + j] = (orc_popcount((unsigned)(i & j)) & 1) ? -r : r;
}

/* The matrix for the head dimension in use, built once and kept (the store
 * and dequant loops would otherwise rebuild it for every slot). */
static const double* orc_hadamard_cached(int D)
{
    static double* H = NULL;
    static int HD = 0;
    if (HD != D) {
        free(H);
        H = (double*)malloc(sizeof(double) * D * D);
        orc_hadamard(D, H);
        HD = D;
    }
    return H;
}

/* ======================================================================
 * Bit packing.  [Atlas] "Background": 3-bit data is 8 values per 3 bytes;
 * 4-bit is two per byte, 2-bit four per byte.  The bit order inside a byte
 * group is not on the pages; the reading used here, for every width b:
 * an LSB-first little-endian bitstream, code i occupying bits
 * [b*i, b*i + b).  At 3 bits this makes every 3-byte group hold 8 whole
 * codes (codes 8g..8g+7 in bytes 3g..3g+2); at 4 bits the low nibble comes
 * first.
 * ==================================================================== */
static void orc_setbit(uint8_t* out, int bit) { out[bit / 8] |= (uint8_t)(1u << (bit % 8)); }
static int orc_getbit(const uint8_t* in, int bit) { return (in[bit / 8] >> (bit % 8)) & 1; }

void orc_pack(const int* codes, int n, int bits, uint8_t* out)
{
    int nbytes = (n * bits + 7) / 8;
    memset(out, 0, (size_t)nbytes);
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < bits; ++j)
            if ((codes[i] >> j) & 1) orc_setbit(out, i * bits + j);
}

void orc_unpack(const uint8_t* in, int n, int bits, int* codes)
{
    for (int i = 0; i < n; ++i) {
        int c = 0;
        for (int j = 0; j < bits; ++j) c |= orc_getbit(in, i * bits + j) << j;
        codes[i] = c;
    }
}

/* ======================================================================
 * Store of one (token, kv head).
 *
 * MSE keys ([vLLM-PR] "implementation breakdown" item 4; [Atlas]
 * "Background"; [vLLM-API] "_store_kv"):
 *   n = ||k||_2;  y = H (s . k) / n;  idx_j = #{midpoints < y_j}
 *   (binary-search bucketize; a value equal to a midpoint takes the lower
 *   index); matched-norm correction stores n / ||c[idx]|| ([Atlas]
 *   "Background": the L2-minimising scale is ||original||/||reconstructed||),
 *   else n; the norm is kept as fp16.  The bucketize decision is taken in
 *   fp32, the precision the midpoints are given in.
 * FP8 keys (k8v4): each coordinate as E4M3, no rotation, no norm.
 * Values ([vLLM-API] "_continuation_prefill" v_scale / v_zero fields):
 *   asymmetric min/max, scale = fp16((max-min)/(2^b-1)), zero = fp16(min),
 *   code = clamp(rint((v - zero)/scale), 0, 2^b-1), all in fp32 with the
 *   fp16-rounded scale and zero; scale == 0 gives code 0 everywhere.
 * ==================================================================== */
static void orc_put_u16(uint8_t* p, uint16_t v)
{
    p[0] = (uint8_t)(v & 0xFF);
    p[1] = (uint8_t)(v >> 8);
}

static uint16_t orc_get_u16(const uint8_t* p)
{
    return (uint16_t)(p[0] | (p[1] << 8));
}

static void orc_store_values(const orc_layout* L, int D, const float* v, uint8_t* slot)
{
    float lo = v[0], hi = v[0];
    for (int i = 1; i < D; ++i) {
        if (v[i] < lo) lo = v[i];
        if (v[i] > hi) hi = v[i];
    }
    const int qmax = (1 << L->value_bits) - 1;
    float range = hi - lo;                           /* one fp32 rounding */
    float scale32 = range / (float)qmax;             /* one fp32 rounding */
    uint16_t scale16 = orc_double_to_f16((double)scale32);
    uint16_t zero16 = orc_double_to_f16((double)lo);
    float sc = (float)orc_f16_to_double(scale16);
    float z = (float)orc_f16_to_double(zero16);
    int* codes = (int*)malloc(sizeof(int) * D);
    for (int i = 0; i < D; ++i) {
        int c = 0;
        if (sc > 0.0f) {
            float t = v[i] - z;
            float u = t / sc;
            float r = nearbyintf(u);
            if (r < 0.0f) r = 0.0f;
            if (r > (float)qmax) r = (float)qmax;
            c = (int)r;
        }
        codes[i] = c;
    }
    orc_pack(codes, D, L->value_bits, slot + L->off_v_data);
    orc_put_u16(slot + L->off_v_scale, scale16);
    orc_put_u16(slot + L->off_v_zero, zero16);
    free(codes);
}

int orc_store_one(int preset, int D, const float* k, const float* v,
                  const int8_t* signs, const float* c32, const float* m32,
                  uint8_t* slot, float* y32)
{
    orc_layout L;
    if (orc_get_layout(preset, D, &L)) return -1;
    memset(slot, 0, (size_t)L.slot_size_aligned);

    if (L.key_fp8) {
        for (int i = 0; i < D; ++i) slot[i] = orc_e4m3_encode((double)k[i]);
    } else {
        const int ncent = 1 << L.key_bits;
        double n2 = 0.0;
        for (int i = 0; i < D; ++i) n2 += (double)k[i] * (double)k[i];
        double n = sqrt(n2);
        const double* H = orc_hadamard_cached(D);
        int* idx = (int*)malloc(sizeof(int) * D);
        double cn2 = 0.0;
        for (int i = 0; i < D; ++i) {
            double r = 0.0;
            for (int j = 0; j < D; ++j) r += H[(size_t)i * D + j] * (signs[j] * (double)k[j]);
            float y = n > 0.0 ? (float)(r / n) : 0.0f;
            if (y32) y32[i] = y;
            int c = 0;
            for (int m = 0; m < ncent - 1; ++m)
                if (m32[m] < y) ++c;
            idx[i] = c;
            cn2 += (double)c32[c] * (double)c32[c];
        }
        double norm = L.norm_correction ? n / sqrt(cn2) : n;
        orc_pack(idx, D, L.key_bits, slot);
        orc_put_u16(slot + L.off_k_norm, orc_double_to_f16(norm));
        free(idx);
    }
    orc_store_values(&L, D, v, slot);
    return 0;
}

/* [vLLM-PR] "turboquant_attn.py": cache (num_blocks, block_size,
 * num_kv_heads, slot); slot index = slot_mapping[token]; block =
 * slot // block_size, offset = slot % block_size.  Negative slots are
 * padding and are not written (the usual vLLM convention). */
/* Where the bytes of slot (block blk, token off, head h) sit in the cache:
 * AoS: one contiguous slot; SoA: a data record and a metadata record.  The
 * copies below move whole slots (in their AoS byte order) in and out. */
static void orc_soa_places(const orc_layout* L, int64_t blk, int bs, int off, int Hk, int h,
                           int64_t* data, int64_t* meta, int* nf, int fields[3])
{
    const int64_t S = L->slot_size_aligned, db = L->key_data_bytes + L->value_data_bytes;
    *nf = L->key_fp8 ? 2 : 3;
    const int64_t rec = (int64_t)off * Hk + h, base = blk * bs * Hk * S;
    *data = base + rec * db;
    *meta = base + (int64_t)bs * Hk * db + rec * 2 * *nf;
    if (L->key_fp8) { fields[0] = L->off_v_scale; fields[1] = L->off_v_zero; }
    else { fields[0] = L->off_k_norm; fields[1] = L->off_v_scale; fields[2] = L->off_v_zero; }
}

static void orc_put_slot(int preset, const orc_layout* L, uint8_t* cache, int64_t blk, int bs,
                         int off, int Hk, int h, const uint8_t* slot)
{
    const int64_t S = L->slot_size_aligned;
    if (!(preset & ORC_LAYOUT_SOA)) {
        memcpy(cache + ((blk * bs + off) * Hk + h) * S, slot, (size_t)S);
        return;
    }
    int64_t data, meta;
    int nf, fields[3];
    orc_soa_places(L, blk, bs, off, Hk, h, &data, &meta, &nf, fields);
    memcpy(cache + data, slot, (size_t)L->key_data_bytes);
    memcpy(cache + data + L->key_data_bytes, slot + L->off_v_data, (size_t)L->value_data_bytes);
    for (int f = 0; f < nf; ++f) memcpy(cache + meta + 2 * f, slot + fields[f], 2);
}

/* The slot's bytes in AoS order: a pointer into the cache (AoS) or `buf`. */
static const uint8_t* orc_get_slot(int preset, const orc_layout* L, const uint8_t* cache, int64_t blk,
                                   int bs, int off, int Hk, int h, uint8_t* buf)
{
    const int64_t S = L->slot_size_aligned;
    if (!(preset & ORC_LAYOUT_SOA)) return cache + ((blk * bs + off) * Hk + h) * S;
    int64_t data, meta;
    int nf, fields[3];
    orc_soa_places(L, blk, bs, off, Hk, h, &data, &meta, &nf, fields);
    memset(buf, 0, (size_t)S);
    memcpy(buf, cache + data, (size_t)L->key_data_bytes);
    memcpy(buf + L->off_v_data, cache + data + L->key_data_bytes, (size_t)L->value_data_bytes);
    for (int f = 0; f < nf; ++f) memcpy(buf + fields[f], cache + meta + 2 * f, 2);
    return buf;
}

int orc_store(int preset, int D, int N, int Hk, int bs,
              const float* key, const float* value, const int64_t* slot_mapping,
              uint8_t* cache, int64_t num_blocks,
              const int8_t* signs, const float* c32, const float* m32)
{
    orc_layout L;
    if (orc_get_layout(preset, D, &L)) return -1;
    const int64_t S = L.slot_size_aligned;
    for (int t = 0; t < N; ++t) {
        int64_t sl = slot_mapping[t];
        if (sl < 0) continue;
        int64_t blk = sl / bs, off = sl % bs;
        if (blk >= num_blocks) return -2;
        for (int h = 0; h < Hk; ++h) {
            uint8_t slot[1024];
            const float* kp = key + ((int64_t)t * Hk + h) * D;
            const float* vp = value + ((int64_t)t * Hk + h) * D;
            if (S > (int64_t)sizeof(slot)) return -1;
            orc_store_one(preset, D, kp, vp, signs, c32, m32, slot, NULL);
            orc_put_slot(preset, &L, cache, blk, bs, (int)off, Hk, h, slot);
        }
    }
    return 0;
}

/* ======================================================================
 * Dequantisation of one slot back to the original space.
 * MSE: y_hat = c[idx]; k_hat = norm * s . (H y_hat)   (H^-1 = H, and the
 * sign flip is its own inverse: [vLLM-API] "_ensure_on_device").
 * FP8: k_hat = E4M3 value.  V: v_hat = code * scale + zero.
 * ==================================================================== */
int orc_dequant_slot(int preset, int D, const uint8_t* slot,
                     const int8_t* signs, const float* c32,
                     double* k_hat, double* v_hat)
{
    orc_layout L;
    if (orc_get_layout(preset, D, &L)) return -1;
    int* codes = (int*)malloc(sizeof(int) * D);
    if (k_hat) {
        if (L.key_fp8) {
            for (int i = 0; i < D; ++i) k_hat[i] = orc_e4m3_decode(slot[i]);
        } else {
            double norm = orc_f16_to_double(orc_get_u16(slot + L.off_k_norm));
            orc_unpack(slot, D, L.key_bits, codes);
            const double* H = orc_hadamard_cached(D);
            for (int i = 0; i < D; ++i) {
                double r = 0.0;
                for (int j = 0; j < D; ++j) r += H[(size_t)i * D + j] * (double)c32[codes[j]];
                k_hat[i] = norm * signs[i] * r;
            }
        }
    }
    if (v_hat) {
        double sc = orc_f16_to_double(orc_get_u16(slot + L.off_v_scale));
        double z = orc_f16_to_double(orc_get_u16(slot + L.off_v_zero));
        orc_unpack(slot + L.off_v_data, D, L.value_bits, codes);
        for (int i = 0; i < D; ++i) v_hat[i] = codes[i] * sc + z;
    }
    free(codes);
    return 0;
}

/* ======================================================================
 * Decode attention.
 *
 * Dense definition ([vLLM-API] "_decode_attention"; paged addressing from
 * [vLLM-PR] "turboquant_attn.py"): for sequence b, token t < seq_len is at
 * page block_table[b][t / bs], offset t % bs.  Query head hq reads kv head
 * hq / (Hq / Hk) ([vLLM-API] "__init__": num_kv_groups).  logits =
 * scale * q . k_hat, softmax over the sequence, out = sum p v_hat,
 * lse = ln sum exp(logit) (natural log, scale included).  An empty
 * sequence gives out = 0 and lse = -inf.
 * ==================================================================== */

int orc_decode_dense(int preset, int D, int B, int Hq, int Hk, int bs,
                     const float* q, const uint8_t* cache, int64_t num_blocks,
                     const int32_t* block_table, int64_t bt_stride,
                     const int32_t* seq_lens, double scale,
                     const int8_t* signs, const float* c32,
                     double* out, double* lse)
{
    orc_layout L;
    if (orc_get_layout(preset, D, &L)) return -1;
    if (Hk <= 0 || Hq % Hk) return -1;
    const int G = Hq / Hk;
    uint8_t sbuf[1024];                      /* a slot gathered from SoA records */
    if (L.slot_size_aligned > (int)sizeof(sbuf)) return -1;
    for (int b = 0; b < B; ++b) {
        const int n = seq_lens[b];
        double* kh = (double*)malloc(sizeof(double) * ((size_t)n * D + 1));
        double* vh = (double*)malloc(sizeof(double) * ((size_t)n * D + 1));
        double* lg = (double*)malloc(sizeof(double) * ((size_t)n + 1));
        for (int h = 0; h < Hk; ++h) {
            for (int t = 0; t < n; ++t) {
                int64_t page = block_table[(int64_t)b * bt_stride + t / bs];
                if (page < 0 || page >= num_blocks) { free(kh); free(vh); free(lg); return -2; }
                orc_dequant_slot(preset, D, orc_get_slot(preset, &L, cache, page, bs, t % bs, Hk, h, sbuf),
                                 signs, c32, kh + (size_t)t * D, vh + (size_t)t * D);
            }
            for (int g = 0; g < G; ++g) {
                const int hq = h * G + g;
                const float* qp = q + ((int64_t)b * Hq + hq) * D;
                double* op = out + ((int64_t)b * Hq + hq) * D;
                for (int i = 0; i < D; ++i) op[i] = 0.0;
                if (n == 0) { lse[(int64_t)b * Hq + hq] = -INFINITY; continue; }
                double m = -INFINITY;
                for (int t = 0; t < n; ++t) {
                    double s = 0.0;
                    for (int i = 0; i < D; ++i) s += (double)qp[i] * kh[(size_t)t * D + i];
                    lg[t] = scale * s;
                    if (lg[t] > m) m = lg[t];
                }
                double den = 0.0;
                for (int t = 0; t < n; ++t) den += exp(lg[t] - m);
                for (int t = 0; t < n; ++t) {
                    double p = exp(lg[t] - m) / den;
                    for (int i = 0; i < D; ++i) op[i] += p * vh[(size_t)t * D + i];
                }
                lse[(int64_t)b * Hq + hq] = m + log(den);
            }
        }
        free(kh); free(vh); free(lg);
    }
    return 0;
}

/* ----------------------------------------------------------------------
 * Split-K form ([vLLM-PR] "implementation breakdown" item 4: stage1 scores
 * and accumulates values per split, stage2 merges by log-sum-exp;
 * [vLLM-PR] "attention.py": the partials carry D values plus one LSE).
 * MSE scores use q rotated once: q . k_hat = norm * <H (s . q), c[idx]>
 * because H is symmetric orthonormal ([Atlas] "weight pre-rotation":
 * <Q H, H K> = <Q, K>).  Split s covers tokens [s*c, min(n, (s+1)*c)) with
 * c = ceil(n / num_splits); empty splits carry lse = -inf and drop out of
 * the merge.
 * -------------------------------------------------------------------- */
int orc_decode_split(int preset, int D, int B, int Hq, int Hk, int bs,
                     const float* q, const uint8_t* cache, int64_t num_blocks,
                     const int32_t* block_table, int64_t bt_stride,
                     const int32_t* seq_lens, double scale, int num_splits,
                     const int8_t* signs, const float* c32,
                     double* out, double* lse)
{
    orc_layout L;
    if (orc_get_layout(preset, D, &L)) return -1;
    if (Hk <= 0 || Hq % Hk || num_splits < 1) return -1;
    const int G = Hq / Hk;
    uint8_t sbuf[1024];                      /* a slot gathered from SoA records */
    if (L.slot_size_aligned > (int)sizeof(sbuf)) return -1;
    double* H = (double*)malloc(sizeof(double) * D * D);
    orc_hadamard(D, H);
    double* qr = (double*)malloc(sizeof(double) * D);
    double* kh = (double*)malloc(sizeof(double) * D);
    double* vh = (double*)malloc(sizeof(double) * D);
    int* codes = (int*)malloc(sizeof(int) * D);
    double* po = (double*)malloc(sizeof(double) * (size_t)num_splits * D);
    double* pl = (double*)malloc(sizeof(double) * (size_t)num_splits);

    for (int b = 0; b < B; ++b) {
        const int n = seq_lens[b];
        const int chunk = (n + num_splits - 1) / num_splits;
        for (int hq = 0; hq < Hq; ++hq) {
            const int h = hq / G;
            const float* qp = q + ((int64_t)b * Hq + hq) * D;
            /* q_rot = H (s . q), once per (b, hq) */
            for (int i = 0; i < D; ++i) {
                double r = 0.0;
                for (int j = 0; j < D; ++j) r += H[(size_t)i * D + j] * (signs[j] * (double)qp[j]);
                qr[i] = r;
            }
            for (int s = 0; s < num_splits; ++s) {
                int t0 = s * chunk, t1 = t0 + chunk;
                if (t1 > n) t1 = n;
                double m = -INFINITY, l = 0.0;
                double* acc = po + (size_t)s * D;
                for (int i = 0; i < D; ++i) acc[i] = 0.0;
                for (int t = t0; t < t1; ++t) {
                    int64_t page = block_table[(int64_t)b * bt_stride + t / bs];
                    if (page < 0 || page >= num_blocks) goto fail;
                    const uint8_t* sp = orc_get_slot(preset, &L, cache, page, bs, t % bs, Hk, h, sbuf);
                    double sc;
                    if (L.key_fp8) {
                        orc_dequant_slot(preset, D, sp, signs, c32, kh, NULL);
                        double d = 0.0;
                        for (int i = 0; i < D; ++i) d += (double)qp[i] * kh[i];
                        sc = scale * d;
                    } else {
                        double norm = orc_f16_to_double(orc_get_u16(sp + L.off_k_norm));
                        orc_unpack(sp, D, L.key_bits, codes);
                        double d = 0.0;
                        for (int i = 0; i < D; ++i) d += qr[i] * (double)c32[codes[i]];
                        sc = scale * norm * d;
                    }
                    orc_dequant_slot(preset, D, sp, signs, c32, NULL, vh);
                    /* online softmax update */
                    double mn = sc > m ? sc : m;
                    double a = exp(m - mn), p = exp(sc - mn);
                    for (int i = 0; i < D; ++i) acc[i] = acc[i] * a + p * vh[i];
                    l = l * a + p;
                    m = mn;
                }
                if (t1 > t0) {
                    for (int i = 0; i < D; ++i) acc[i] /= l;
                    pl[s] = m + log(l);
                } else {
                    pl[s] = -INFINITY;
                }
            }
            /* stage2: log-sum-exp merge */
            double M = -INFINITY;
            for (int s = 0; s < num_splits; ++s) if (pl[s] > M) M = pl[s];
            double* op = out + ((int64_t)b * Hq + hq) * D;
            for (int i = 0; i < D; ++i) op[i] = 0.0;
            if (M == -INFINITY) { lse[(int64_t)b * Hq + hq] = -INFINITY; continue; }
            double W = 0.0;
            for (int s = 0; s < num_splits; ++s) {
                if (pl[s] == -INFINITY) continue;
                double w = exp(pl[s] - M);
                W += w;
                for (int i = 0; i < D; ++i) op[i] += w * po[(size_t)s * D + i];
            }
            for (int i = 0; i < D; ++i) op[i] /= W;
            lse[(int64_t)b * Hq + hq] = M + log(W);
        }
    }
    free(H); free(qr); free(kh); free(vh); free(codes); free(po); free(pl);
    return 0;
fail:
    free(H); free(qr); free(kh); free(vh); free(codes); free(po); free(pl);
    return -2;
}

int orc_sparse_v_bound(int preset, int D, int B, int Hq, int Hk, int bs,
                       const float* q, const uint8_t* cache, int64_t num_blocks,
                       const int32_t* block_table, int64_t bt_stride,
                       const int32_t* seq_lens, double scale, double tau,
                       const int8_t* signs, const float* c32,
                       double* bound, double* mass)
{
    orc_layout L;
    if (orc_get_layout(preset, D, &L)) return -1;
    if (Hk <= 0 || Hq % Hk) return -1;
    const int G = Hq / Hk;
    uint8_t sbuf[1024];                      /* a slot gathered from SoA records */
    if (L.slot_size_aligned > (int)sizeof(sbuf)) return -1;
    for (int b = 0; b < B; ++b) {
        const int n = seq_lens[b];
        double* kh = (double*)malloc(sizeof(double) * ((size_t)n * D + 1));
        double* vh = (double*)malloc(sizeof(double) * ((size_t)n * D + 1));
        double* lg = (double*)malloc(sizeof(double) * ((size_t)n + 1));
        for (int h = 0; h < Hk; ++h) {
            for (int t = 0; t < n; ++t) {
                int64_t page = block_table[(int64_t)b * bt_stride + t / bs];
                if (page < 0 || page >= num_blocks) { free(kh); free(vh); free(lg); return -2; }
                orc_dequant_slot(preset, D, orc_get_slot(preset, &L, cache, page, bs, t % bs, Hk, h, sbuf),
                                 signs, c32, kh + (size_t)t * D, vh + (size_t)t * D);
            }
            for (int g = 0; g < G; ++g) {
                const int hq = h * G + g;
                const float* qp = q + ((int64_t)b * Hq + hq) * D;
                double* bp = bound + ((int64_t)b * Hq + hq) * D;
                for (int i = 0; i < D; ++i) bp[i] = 0.0;
                mass[(int64_t)b * Hq + hq] = 0.0;
                if (n == 0) continue;
                double m = -INFINITY;
                for (int t = 0; t < n; ++t) {
                    double s = 0.0;
                    for (int i = 0; i < D; ++i) s += (double)qp[i] * kh[(size_t)t * D + i];
                    lg[t] = scale * s;
                    if (lg[t] > m) m = lg[t];
                }
                double den = 0.0, dropped = 0.0;
                for (int t = 0; t < n; ++t) den += exp(lg[t] - m);
                for (int t = 0; t < n; ++t) {
                    const double e = exp(lg[t] - m);
                    if (e > tau) continue;
                    dropped += e;
                    for (int i = 0; i < D; ++i) bp[i] += e * fabs(vh[(size_t)t * D + i]);
                }
                for (int i = 0; i < D; ++i) bp[i] /= den;
                mass[(int64_t)b * Hq + hq] = dropped / den;
            }
        }
        free(kh); free(vh); free(lg);
    }
    return 0;
}
