"""Float64 CPU oracle (test infrastructure; see mla_oracle's module docstring)."""
