"""GB300-native absorbed MLA decode over a paged latent cache (placeholder; binding follows)."""
