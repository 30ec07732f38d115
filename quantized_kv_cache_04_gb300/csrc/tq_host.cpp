// Host side of the TurboQuant C ABI: slot layout, Lloyd-Max codebook,
// Rademacher signs, split heuristic, workspace sizing and status strings.
// Nothing here touches the GPU.
#include "tq.h"
#include "tq_internal.h"

#include <cmath>
#include <cstring>
#include <vector>

namespace tq {

int fill_layout(int preset, int head_dim, tq_layout* L)
{
    if (!L || head_dim <= 0 || head_dim % 8) return TQ_ERR_INVALID_ARG;
    if (!layout_flags_ok(preset)) return TQ_ERR_UNSUPPORTED;
    preset &= 0xFF;                    // the block convention does not change the slot
    std::memset(L, 0, sizeof(*L));
    // Preset table: "turboquant_attn.py" supported_kv_cache_dtypes; key/value
    // widths as the preset names spell them (k8 = FP8 keys, v4 = 4-bit values,
    // _nc = norm correction).
    switch (preset) {
    case TQ_K8V4:    L->key_fp8 = 1; L->key_bits = 8; L->value_bits = 4; L->norm_correction = 0; break;
    case TQ_4BIT_NC: L->key_bits = 4; L->value_bits = 4; L->norm_correction = 1; break;
    case TQ_K3V4_NC: L->key_bits = 3; L->value_bits = 4; L->norm_correction = 1; break;
    case TQ_3BIT_NC: L->key_bits = 3; L->value_bits = 3; L->norm_correction = 1; break;
    case TQ_2BIT_NC: L->key_bits = 2; L->value_bits = 2; L->norm_correction = 1; break;
    default: return TQ_ERR_UNSUPPORTED;
    }
    const int D = head_dim;
    L->n_centroids = L->key_fp8 ? 0 : (1 << L->key_bits);
    L->key_data_bytes = L->key_fp8 ? D : (D * L->key_bits + 7) / 8;
    L->off_k_norm = L->key_fp8 ? -1 : L->key_data_bytes;
    L->key_packed_size = L->key_data_bytes + (L->key_fp8 ? 0 : 2);
    L->value_data_bytes = (D * L->value_bits + 7) / 8;
    L->off_v_data = L->key_packed_size;
    L->off_v_scale = L->off_v_data + L->value_data_bytes;
    L->off_v_zero = L->off_v_scale + 2;
    L->value_packed_size = L->value_data_bytes + 4;
    L->slot_size = L->key_packed_size + L->value_packed_size;
    L->slot_size_aligned = (L->slot_size + 1) & ~1;
    return TQ_OK;
}

}  // namespace tq

extern "C" int tq_get_layout(int preset, int head_dim, tq_layout* out)
{
    return tq::fill_layout(preset, head_dim, out);
}

// Lloyd-Max scalar quantizer for N(0, 1/d), following the solve_lloyd_max
// steps of the "centroids.py" section: uniform-cell init on +-3.5 sigma,
// boundaries = neighbour means with outer edges at +-10.5 sigma, centroid =
// cell mass-weighted mean by 200-panel trapezoid sums, stop when no centroid
// moves by 1e-10 or more (keeping the iterate that did not move), else after
// 200 rounds.
extern "C" int tq_build_codebook(int head_dim, int bits, float* centroids, float* midpoints)
{
    if (head_dim <= 0 || bits < 1 || bits > 8 || !centroids) return TQ_ERR_INVALID_ARG;
    const int levels = 1 << bits, panels = 200, rounds = 200;
    const double var = 1.0 / head_dim, sd = std::sqrt(var);
    const double lo = -3.5 * sd, hi = 3.5 * sd;
    const double norm_const = 1.0 / std::sqrt(2 * M_PI * var);
    auto density = [&](double x) { return norm_const * std::exp(-x * x / (2 * var)); };

    std::vector<double> cur(levels), next(levels), edge(levels + 1);
    for (int i = 0; i < levels; ++i) cur[i] = lo + (hi - lo) * (i + 0.5) / levels;
    for (int r = 0; r < rounds; ++r) {
        edge.front() = lo * 3;
        edge.back() = hi * 3;
        for (int i = 1; i < levels; ++i) edge[i] = (cur[i - 1] + cur[i]) / 2.0;
        double largest_move = 0.0;
        for (int i = 0; i < levels; ++i) {
            const double a = edge[i], b = edge[i + 1], h = (b - a) / panels;
            const double da = density(a), db = density(b);
            double mass = 0.5 * (da + db), moment = 0.5 * (a * da + b * db);
            for (int p = 1; p < panels; ++p) {
                const double x = a + p * h, f = density(x);
                mass += f;
                moment += x * f;
            }
            mass *= h;
            moment *= h;
            next[i] = mass > 1e-15 ? moment / mass : cur[i];
            largest_move = std::fmax(largest_move, std::fabs(next[i] - cur[i]));
        }
        if (largest_move < 1e-10) break;
        cur.swap(next);
    }
    for (int i = 0; i < levels; ++i) centroids[i] = static_cast<float>(cur[i]);
    if (midpoints)
        for (int i = 0; i + 1 < levels; ++i) midpoints[i] = (centroids[i] + centroids[i + 1]) / 2.0f;
    return TQ_OK;
}

// SplitMix64 (Steele, Lea & Flood 2014): output i of the generator whose
// state starts at `seed` is the finaliser applied to seed + (i+1)*golden.
extern "C" int tq_make_signs(int head_dim, uint64_t seed, int8_t* signs)
{
    if (head_dim <= 0 || !signs) return TQ_ERR_INVALID_ARG;
    uint64_t state = seed;
    for (int i = 0; i < head_dim; ++i) {
        state += 0x9E3779B97F4A7C15ULL;
        uint64_t z = state;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
        z ^= z >> 31;
        signs[i] = (z >> 63) ? int8_t(-1) : int8_t(1);
    }
    return TQ_OK;
}

extern "C" size_t tq_decode_workspace_bytes(int batch, int num_q_heads, int num_splits, int head_dim)
{
    if (batch <= 0 || num_q_heads <= 0 || num_splits <= 0 || head_dim <= 0) return 0;
    return (size_t)batch * num_q_heads * num_splits * (head_dim + 1) * sizeof(float);
}

extern "C" int tq_decode_pick_splits(int preset, int head_dim, int batch, int num_q_heads,
                                     int num_kv_heads, int max_seq_len)
{
    tq_layout L;
    const int rc = tq::fill_layout(preset, head_dim, &L);
    if (rc) return rc;
    if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads) return TQ_ERR_INVALID_ARG;
    return tq::pick_splits(L, tq::is_soa(preset), batch, num_q_heads, num_kv_heads, max_seq_len);
}

extern "C" const char* tq_status_string(int status)
{
    switch (status) {
    case TQ_OK: return "ok";
    case TQ_ERR_INVALID_ARG: return "invalid argument (null pointer or bad size)";
    case TQ_ERR_UNSUPPORTED: return "unsupported preset, head_dim, block_size or dtype";
    case TQ_ERR_WORKSPACE: return "workspace too small (see tq_decode_workspace_bytes)";
    case TQ_ERR_CUDA: return "CUDA launch or device error";
    default: return "unknown status";
    }
}

extern "C" int tq_version(void) { return 100; }
