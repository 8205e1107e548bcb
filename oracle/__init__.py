"""Float64 CPU oracle (test infrastructure only; see ``bsattn_oracle``)."""
