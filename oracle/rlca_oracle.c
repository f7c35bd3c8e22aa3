/*
 * Oracle for RL credit assignment: plain, slow, obviously correct reverse loops in fp64.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's CPU
 * baseline use this file. It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (source: "rl-triton: High-Performance Triton GPU Kernels for
 * Reinforcement Learning Credit Assignment", technical summary):
 *   - Problem statement: credit-assignment quantities over [num_envs, seq_len] tensors of
 *     rewards, values and done flags, each a first-order linear recurrence in time.
 *   - Method section 1 (unified algebraic framework): every estimator is an instance of
 *     A_t = alpha_t + beta_t * A_{t+1}. This oracle does NOT use that form; it writes each
 *     estimator's textbook recursion out directly, one env at a time, t = T-1 down to 0.
 *   - Method section 3 (explicit boundary semantics): a terminated step has successor
 *     value 0; a truncated step uses a supplied bootstrap value; the last step of the
 *     rollout window (t = T-1) bootstraps from the supplied per-env value. The bootstrap
 *     enters the last step's own update, never a separate scan carry, so it is counted
 *     once.
 * The pages print no per-estimator formula. The definitions used are the textbook ones:
 * discounted return; GAE (Schulman et al. 2016); TD(lambda) lambda-returns (Sutton &
 * Barto); V-trace (Espeholt et al. 2018, IMPALA, with lambda on the trace coefficient);
 * Retrace(lambda) (Munos et al. 2016).
 *
 * Readings where the pages are silent:
 *   - terminated and truncated at the same step: termination wins (successor value 0);
 *   - truncated at t = T-1: the truncation value wins over the window bootstrap;
 *   - bootstrap == NULL means 0; truncated == NULL means no truncation;
 *   - trunc_value is read only where truncated is set.
 *
 * Layout: inputs are row-major [N, ld] (T <= ld used per row); per-env bootstrap is [N];
 * outputs are dense row-major [N, T] doubles. Flags are bytes, nonzero = set.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

/* Value of the state after step t of row n, as the boundary rules define it. */
static double successor_value(const uint8_t *term, const uint8_t *trunc, const float *tv,
                              const float *boot, const float *next_row_value,
                              int64_t n, int64_t t, int64_t T, int64_t i)
{
    if (term[i]) return 0.0;
    if (trunc && trunc[i]) return (double)tv[i];
    if (t == T - 1) return boot ? (double)boot[n] : 0.0;
    return (double)next_row_value[i + 1];
}

/* True when no credit flows from step t+1 into step t: the episode ended at t
 * (terminated or truncated) or t is the last step of the window. */
static int stops(const uint8_t *term, const uint8_t *trunc, int64_t t, int64_t T, int64_t i)
{
    return term[i] || (trunc && trunc[i]) || t == T - 1;
}

/* Discounted return: G_t = r_t + gamma * (successor value, or G_{t+1} inside an episode). */
void oracle_discounted_return(const float *reward, const uint8_t *term, const uint8_t *trunc,
                              const float *tv, const float *boot, double gamma,
                              int64_t N, int64_t T, int64_t ld, double *ret)
{
    for (int64_t n = 0; n < N; ++n) {
        double g_next = 0.0;
        for (int64_t t = T - 1; t >= 0; --t) {
            int64_t i = n * ld + t;
            double next;
            if (term[i]) next = 0.0;
            else if (trunc && trunc[i]) next = (double)tv[i];
            else if (t == T - 1) next = boot ? (double)boot[n] : 0.0;
            else next = g_next;
            double g = (double)reward[i] + gamma * next;
            ret[n * T + t] = g;
            g_next = g;
        }
    }
}

/* GAE: delta_t = r_t + gamma * V(s_{t+1}) - V_t, A_t = delta_t + gamma*lambda*A_{t+1}
 * inside an episode, A_t = delta_t at its last step; returns_t = A_t + V_t. */
void oracle_gae(const float *reward, const float *value, const uint8_t *term,
                const uint8_t *trunc, const float *tv, const float *boot, double gamma,
                double lambda, int64_t N, int64_t T, int64_t ld, double *adv, double *ret)
{
    for (int64_t n = 0; n < N; ++n) {
        double a_next = 0.0;
        for (int64_t t = T - 1; t >= 0; --t) {
            int64_t i = n * ld + t;
            double nv = successor_value(term, trunc, tv, boot, value, n, t, T, i);
            double v = (double)value[i];
            double delta = (double)reward[i] + gamma * nv - v;
            double a = stops(term, trunc, t, T, i) ? delta : delta + gamma * lambda * a_next;
            adv[n * T + t] = a;
            if (ret) ret[n * T + t] = a + v;
            a_next = a;
        }
    }
}

/* TD(lambda) lambda-return: G_t = r_t + gamma * ((1-lambda) V_{t+1} + lambda G_{t+1})
 * inside an episode, G_t = r_t + gamma * (successor value) at its last step. */
void oracle_td_lambda(const float *reward, const float *value, const uint8_t *term,
                      const uint8_t *trunc, const float *tv, const float *boot, double gamma,
                      double lambda, int64_t N, int64_t T, int64_t ld, double *target)
{
    for (int64_t n = 0; n < N; ++n) {
        double g_next = 0.0;
        for (int64_t t = T - 1; t >= 0; --t) {
            int64_t i = n * ld + t;
            double g;
            if (stops(term, trunc, t, T, i)) {
                g = (double)reward[i]
                    + gamma * successor_value(term, trunc, tv, boot, value, n, t, T, i);
            } else {
                g = (double)reward[i]
                    + gamma * ((1.0 - lambda) * (double)value[i + 1] + lambda * g_next);
            }
            target[n * T + t] = g;
            g_next = g;
        }
    }
}

/* V-trace (IMPALA): with rho_t = exp(log_rho_t), rho_hat_t = min(rho_bar, rho_t),
 * c_t = lambda * min(c_bar, rho_t),
 *   vs_t - V_t = rho_hat_t (r_t + gamma V(s_{t+1}) - V_t) + gamma c_t (vs_{t+1} - V_{t+1})
 * inside an episode (the second term is absent at its last step), and the policy-gradient
 * advantage pg_t = min(pg_rho_bar, rho_t) (r_t + gamma q_{t+1} - V_t), where q_{t+1} is
 * vs_{t+1} inside an episode and the successor value at its last step. */
void oracle_vtrace(const float *reward, const float *value, const float *log_rho,
                   const uint8_t *term, const uint8_t *trunc, const float *tv,
                   const float *boot, double gamma, double lambda, double rho_bar,
                   double c_bar, double pg_rho_bar, int64_t N, int64_t T, int64_t ld,
                   double *vs, double *pg)
{
    for (int64_t n = 0; n < N; ++n) {
        double vs_next = 0.0, v_next = 0.0;
        for (int64_t t = T - 1; t >= 0; --t) {
            int64_t i = n * ld + t;
            double rho = exp((double)log_rho[i]);
            double rho_hat = rho < rho_bar ? rho : rho_bar;
            double c = lambda * (rho < c_bar ? rho : c_bar);
            double v = (double)value[i];
            double nv = successor_value(term, trunc, tv, boot, value, n, t, T, i);
            int stop = stops(term, trunc, t, T, i);
            double diff = rho_hat * ((double)reward[i] + gamma * nv - v);
            if (!stop) diff += gamma * c * (vs_next - v_next);
            double vs_t = v + diff;
            vs[n * T + t] = vs_t;
            if (pg) {
                double rho_pg = rho < pg_rho_bar ? rho : pg_rho_bar;
                double q = stop ? nv : vs_next;
                pg[n * T + t] = rho_pg * ((double)reward[i] + gamma * q - v);
            }
            vs_next = vs_t;
            v_next = v;
        }
    }
}

/* Retrace(lambda): with c_t = lambda * min(1, rho_t),
 *   Q^ret_t = r_t + gamma E_pi Q(s_{t+1},.) + gamma c_{t+1} (Q^ret_{t+1} - Q(s_{t+1},a_{t+1}))
 * inside an episode (the last term is absent at its last step). E_pi Q(s_{t+1},.) is
 * expected_q[t+1] inside an episode; at its last step it is 0 if terminated, the
 * truncation value if truncated, else the per-env window bootstrap. */
void oracle_retrace(const float *reward, const float *q_taken, const float *expected_q,
                    const float *rho, const uint8_t *term, const uint8_t *trunc,
                    const float *tv, const float *boot_ev, double gamma, double lambda,
                    int64_t N, int64_t T, int64_t ld, double *q_ret)
{
    for (int64_t n = 0; n < N; ++n) {
        double qret_next = 0.0;
        for (int64_t t = T - 1; t >= 0; --t) {
            int64_t i = n * ld + t;
            double nev = successor_value(term, trunc, tv, boot_ev, expected_q, n, t, T, i);
            double q = (double)reward[i] + gamma * nev;
            if (!stops(term, trunc, t, T, i)) {
                double rho1 = (double)rho[i + 1];
                double c1 = lambda * (rho1 < 1.0 ? rho1 : 1.0);
                q += gamma * c1 * (qret_next - (double)q_taken[i + 1]);
            }
            q_ret[n * T + t] = q;
            qret_next = q;
        }
    }
}

/* ------------------------------------------------------------------ forward scans
 * The forward-time mirror of the recurrence (Method section 1: eligibility traces run
 * the same first-order recurrence forward in time; episodic prefix sums are its decay-1
 * case): A_t = x_t + decay * A_{t-1} inside an episode. A step that follows the end of
 * an episode (the previous step terminated or truncated) starts afresh: A_t = x_t. At
 * the window start A_{-1} is the per-env carried-in value init[n] (NULL means 0), the
 * forward counterpart of the window-end bootstrap (Method section 3). */

/* Accumulating eligibility trace e_t = x_t + decay * e_{t-1} (decay = gamma * lambda). */
void oracle_eligibility_trace(const float *x, const uint8_t *term, const uint8_t *trunc,
                              const float *init, double decay, int64_t N, int64_t T,
                              int64_t ld, double *trace)
{
    for (int64_t n = 0; n < N; ++n) {
        double prev = init ? (double)init[n] : 0.0;
        for (int64_t t = 0; t < T; ++t) {
            int64_t i = n * ld + t;
            int fresh = t > 0 && (term[i - 1] || (trunc && trunc[i - 1]));
            double e = fresh ? (double)x[i] : (double)x[i] + decay * prev;
            trace[n * T + t] = e;
            prev = e;
        }
    }
}

/* Episodic prefix sum S_t = x_t + S_{t-1} inside an episode. */
void oracle_episodic_prefix_sum(const float *x, const uint8_t *term, const uint8_t *trunc,
                                const float *init, int64_t N, int64_t T, int64_t ld,
                                double *sum)
{
    for (int64_t n = 0; n < N; ++n) {
        double prev = init ? (double)init[n] : 0.0;
        for (int64_t t = 0; t < T; ++t) {
            int64_t i = n * ld + t;
            int fresh = t > 0 && (term[i - 1] || (trunc && trunc[i - 1]));
            double s = fresh ? (double)x[i] : (double)x[i] + prev;
            sum[n * T + t] = s;
            prev = s;
        }
    }
}
