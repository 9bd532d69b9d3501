// Critical-wave model constants used when a plan leaves the model parameters
// at their defaults (LiquidCP Section 5.2, Eqs. 5-6; Appendix A.2
// "Calibration").  Written by long_context_split_gb300/calibrate.py on 2026-12-02
// (NVIDIA GB300); a kernel without a fit keeps LiquidCP Table 2's H100 values.
#pragma once

namespace skv {
namespace calib {

struct Fit {
    double rho, delta_attn, delta_red, gamma;
};

constexpr Fit kGqaEngine = {1.0, 0.0, 2.5, 2.0};   // time unit 0.836 us per tile-equivalent, relative RMS error 3.2 %
constexpr Fit kMla = {1.0, 8.0, 1.0, 0.0};   // time unit 2.251 us per tile-equivalent, relative RMS error 2.8 %
constexpr Fit kTable2 = {0.43, 32.0, 2.5, 0.47};

}  // namespace calib
}  // namespace skv
