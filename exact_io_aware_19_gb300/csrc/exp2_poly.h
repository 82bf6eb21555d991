// exp2_poly.h — written by exact_io_aware_19_gb300/fit_exp2_poly.py; do not edit.
// Degree-3 minimax fit of 2^f on [-1/2, 1/2] (relative error), fp32 coefficients.
// LP optimum 7.477e-05; measured with fp32 Horner evaluation: 7.485e-05.
#pragma once

namespace ex19 {
constexpr float kExp2PolyMaxRelErr = 7.485e-05f;
constexpr float kExp2C0 = 0.9999280571937561f;
constexpr float kExp2C1 = 0.6932608485221863f;
constexpr float kExp2C2 = 0.24261115491390228f;
constexpr float kExp2C3 = 0.05517221987247467f;
}  // namespace ex19
