"""GB300 (sm_103a) decode-time Multi-matrix Factorization Attention (MFA)."""
