"""fp8 e4m3 latent-KV absorbed MLA decode for one GB300 (sm_103a)."""
