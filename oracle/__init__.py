"""Float64 CPU oracle of scaled dot-product attention.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU legs (CPU baseline, reference arm), never by the library.
"""
from .sdpa_oracle import (  # noqa: F401
    Band, Dropout, band_bias, causal_bias, default_scale, dropout_keep, gather_paged, philox4x32_10, ref_backward,
    ref_forward, ref_forward_paged, ref_forward_rows, ref_backward_rows, ref_group,
)
