"""Paged Gated Delta-Rule (GDN) prefill and decode for GB300 (sm_103a)."""
