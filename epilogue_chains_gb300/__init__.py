"""epilogue_chains_gb300: vertical fusion of dependent operator chains on one GB300 (sm_103a)."""
